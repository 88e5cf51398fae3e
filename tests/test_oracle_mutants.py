"""The pins must be sensitive: plant plausible mistakes in a copy of the
oracle's C source, build it, and check that at least one pin fails for each.

The mistakes are planted on the CPU, in a temporary copy; the committed
oracle is untouched.
"""
import os
import shutil
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "oracle.c")

# (name, text in oracle.c, replacement)
MUTANTS = [
    ("dropped 1/sqrt2 in phi", "x[a] * x[b] * inv_sqrt2", "x[a] * x[b]"),
    ("column-major quadratic block", "phi[1 + dfeat + a * dfeat + b] = x[a] * x[b] * inv_sqrt2",
     "phi[1 + dfeat + a * dfeat + b] = x[a] * x[(b + 1) % dfeat] * inv_sqrt2"),
    ("normaliser not accumulated", "z[r] = lam * z[r] + phk[r];", "z[r] = phk[r];"),
    ("decay applied after the write", "s[r * dv + c] = lam * s[r * dv + c] + phk[r] * vt[c];",
     "s[r * dv + c] = lam * (s[r * dv + c] + phk[r] * vt[c]);"),
    ("decay skipped on the normaliser", "z[r] = lam * z[r] + phk[r];", "z[r] = z[r] + phk[r];"),
    ("eps forced to one", "y[c] = nm / (dn + j->eps);", "y[c] = nm / (dn + 1.0);"),
    ("delta-rule sign flipped", "al * (S[i * dk + a] - be * Sk[i] * kt[a])", "al * (S[i * dk + a] + be * Sk[i] * kt[a])"),
    ("write decayed by alpha", "+ be * vt[i] * kt[a];", "+ al * be * vt[i] * kt[a];"),
    ("beta dropped from erase", "al * (S[i * dk + a] - be * Sk[i] * kt[a])", "al * (S[i * dk + a] - Sk[i] * kt[a])"),
    ("query read with the key", "acc += S[i * dk + a] * qt[a];", "acc += S[i * dk + a] * kt[a];"),
    ("state_in ignored", "S[i] = j->s_in ? j->s_in[bh * dv * dk + i] : 0.0;", "S[i] = 0.0;"),
    ("scalar gate: decay dropped", "S[i * dk + a] = al * S[i * dk + a] + be * vt[i] * kt[a];",
     "S[i * dk + a] = S[i * dk + a] + be * vt[i] * kt[a];"),
    ("scalar gate: write decayed", "S[i * dk + a] = al * S[i * dk + a] + be * vt[i] * kt[a];",
     "S[i * dk + a] = al * (S[i * dk + a] + be * vt[i] * kt[a]);"),
    ("scalar gate: beta dropped", "S[i * dk + a] = al * S[i * dk + a] + be * vt[i] * kt[a];",
     "S[i * dk + a] = al * S[i * dk + a] + vt[i] * kt[a];"),
]

PIN_FUNCS = [
    lambda: pins.test_feature_inner_product_is_closed_form_kernel(4),
    pins.test_feature_layout_row_major_and_constant_term,
    lambda: pins.test_taylor_equals_quadratic_form(4, 5, 37),
    pins.test_taylor_state_invariants,
    pins.test_taylor_zero_query_is_running_mean,
    lambda: pins.test_taylor_decay_equals_weighted_quadratic_form(4, 5, 33),
    pins.test_taylor_decay_split_resume_with_state,
    lambda: pins.test_gdn_equals_dense_matrix_form(6, 5, 23),
    pins.test_gdn_reduces_to_additive_for_orthogonal_keys,
    pins.test_gdn_beta_zero_pure_decay,
    pins.test_gdn_overwrite_property_unit_keys,
    pins.test_gdn_q_scale_split_and_samples,
    lambda: pins.test_gated_equals_closed_form(6, 5, 17),
    pins.test_gated_equals_delta_rule_for_orthogonal_keys,
    pins.test_gated_additive_special_case,
]


def _caught(fn) -> bool:
    try:
        fn()
    except AssertionError:
        return True
    return False


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    text = open(SRC).read()
    assert old in text, f"mutation anchor for '{name}' not found in oracle.c"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new, 1))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-std=c11", "-o", str(so), str(src), "-lm"],
                   check=True)
    oracle._load()
    prev = oracle.load_library(str(so))
    try:
        caught = [_caught(f) for f in PIN_FUNCS]
    finally:
        oracle.restore_library(prev)
    assert any(caught), f"no pin caught the planted mistake '{name}'"


# Planted mistakes in the numpy definitions (the NoteBank write side and routing): the function is
# rebuilt from an edited copy of its source and swapped in while the NoteBank pins run.
PY_SRC = os.path.join(os.path.dirname(SRC), "__init__.py")
PY_MUTANTS = [
    ("chunk mean not re-normalised", "mu = _unit(kh[:, :, c0:c1].mean(axis=2))", "mu = kh[:, :, c0:c1].mean(axis=2)"),
    ("keys not normalised", "kh = _unit(k)", "kh = k"),
    ("window one token short", "w = np.array([d[t:t + window].sum()", "w = np.array([d[t:t + window - 1].sum()"),
    ("channel mean over tokens", "d = d_ch.mean(axis=(0, 1))", "d = d_ch.mean(axis=(0, 1)) * 0 + d_ch.mean()"),
    ("last maximum on ties", "t = int(s0 + int(np.argmax(seg)))",
     "t = int(s0 + len(seg) - 1 - int(np.argmax(seg[::-1])))"),
    ("address gathered at the span start", "rho[i, l, h] = _round_bf16(qf[l, h, t,", "rho[i, l, h] = _round_bf16(qf[l, h, s0,"),
    ("later note wins equal votes", "key=lambda i: (-votes[i], i))[:R]", "key=lambda i: (-votes[i], -i))[:R]"),
    ("retrieved in vote order", "top = np.array(sorted(order, key=lambda i: (pos[i], i)), dtype=np.int64)",
     "top = np.array(order, dtype=np.int64)"),
    ("mean instead of max over the question", "s[:, j] = np.max(rn[:, j, :] @ un[j].T, axis=1)",
     "s[:, j] = np.mean(rn[:, j, :] @ un[j].T, axis=1)"),
]
NB_PINS = [pins.test_notebank_scores_hand_example, pins.test_notebank_scores_identities,
           pins.test_notebank_address_argmax_and_gather, pins.test_notebank_route_worked_example,
           pins.test_notebank_route_ties_scaling_and_max_over_question]


@pytest.mark.parametrize("name,old,new", PY_MUTANTS, ids=[m[0] for m in PY_MUTANTS])
def test_notebank_pins_catch_planted_mistake(monkeypatch, name, old, new):
    text = open(PY_SRC).read()
    assert old in text, f"mutation anchor for '{name}' not found"
    ns = {"__name__": "oracle_mutant", "__file__": PY_SRC}
    exec(compile(text.replace(old, new, 1), "oracle_mutant", "exec"), ns)
    for fn in ("notebank_scores", "notebank_address", "notebank_route"):
        monkeypatch.setattr(oracle, fn, ns[fn])
    assert any(_caught(f) for f in NB_PINS), f"no pin caught the planted mistake '{name}'"


# Planted mistakes in the window-attention and state-operation definitions, against their pins.
SWA_STATE_MUTANTS = [
    ("window one token too long", "lo = max(0, i - window + 1)", "lo = max(0, i - window)"),
    ("window excludes the current token", "for j in range(lo, i + 1)])", "for j in range(lo, i)] + [0.0])"),
    ("scale dropped", "s = np.array([scale * float(np.dot(q[b, h, i], k[b, h, j]))",
     "s = np.array([float(np.dot(q[b, h, i], k[b, h, j]))"),
    ("softmax not normalised", "/ e.sum()", "/ 1.0"),
    ("reset keeps the state", "np.zeros_like(x[idx]) if lam[idx] == 0 else", "x[idx] if lam[idx] == 0 else"),
    ("rescale by lambda squared", "(lam[idx] * x[idx]).astype(np.float32)", "(lam[idx] * lam[idx] * x[idx]).astype(np.float32)"),
    ("gather reads the next state", "np.stack([flat[int(i)].copy() for i in index])",
     "np.stack([flat[(int(i) + 1) % len(flat)].copy() for i in index])"),
]
SWA_STATE_PINS = [lambda: pins.test_swa_equals_banded_matrix_softmax(5), lambda: pins.test_swa_equals_banded_matrix_softmax(1),
                  pins.test_swa_special_cases, pins.test_state_rescale_definition_and_reset,
                  pins.test_state_rescale_feeds_the_recurrence_linearly, pins.test_state_gather_copies_and_branches]


@pytest.mark.parametrize("name,old,new", SWA_STATE_MUTANTS, ids=[m[0] for m in SWA_STATE_MUTANTS])
def test_window_and_state_pins_catch_planted_mistake(monkeypatch, name, old, new):
    text = open(PY_SRC).read()
    assert old in text, f"mutation anchor for '{name}' not found"
    ns = {"__name__": "oracle_mutant", "__file__": PY_SRC}
    exec(compile(text.replace(old, new, 1), "oracle_mutant", "exec"), ns)
    for fn in ("swa", "state_rescale", "state_gather"):
        monkeypatch.setattr(oracle, fn, ns[fn])
    assert any(_caught(f) for f in SWA_STATE_PINS), f"no pin caught the planted mistake '{name}'"
