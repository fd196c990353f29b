"""The pins must catch plausible mistakes in the oracle (CPU only).

Each case copies ``oracle/delta_oracle.c`` to a temporary directory, plants
ONE mistake by a textual edit, compiles the copy and runs every pin in
``pins.py`` against it: at least one pin has to fail.  The oracle's own
source is never modified.
"""
import functools
import os
import subprocess

import numpy as np
import pytest

import oracle
from pins import ALL_CHECKS

SRC = os.path.join(os.path.dirname(oracle.__file__), "delta_oracle.c")

READOUT = """        /* out_t = S^T q_t, after the token's update */
        const float *qq = J->q + ((b * T + t) * H + h) * dk;
        double *oo = J->out + ((b * T + t) * H + h) * dv;
        for (int64_t c = 0; c < dv; ++c) {
            double acc = 0.0;
            for (int64_t d = 0; d < dk; ++d) acc += S[d * dv + c] * (double)qq[d];
            oo[c] = acc;
        }
"""
GATE = """        if (J->g) {
            const double gt = (double)J->g[(b * T + t) * H + h];
            for (int64_t i = 0; i < dk * dv; ++i) S[i] *= gt;
        }
"""
SUBSTEP_HEAD = "        for (int64_t j = 0; j < n_h; ++j) {\n"

MUTANTS = {
    # a wrong sign on the write
    "write_sign": [("S[d * dv + c] += s * e[c];", "S[d * dv + c] -= s * e[c];")],
    # a wrong sign inside the prediction error
    "error_sign": [("e[c] = (double)vv[c] - acc;", "e[c] = acc - (double)vv[c];")],
    # a dropped term: write v instead of the residual (Hebbian, no erase)
    "no_erase": [("e[c] = (double)vv[c] - acc;", "e[c] = (double)vv[c] + 0.0 * acc;")],
    # beta dropped (treated as 1)
    "no_beta": [("const double bb = (double)J->beta[row];", "const double bb = 1.0;")],
    # readout taken before the token's update
    "readout_before_update": [(GATE, READOUT.replace("\n", "\n", 1) + GATE),
                              ("    }\n\n    if (J->hT) {", "    }\n\n    if (J->hT) {")],
    # the sub-steps run in reverse order
    "substeps_reversed": [(SUBSTEP_HEAD,
                           "        for (int64_t j = n_h - 1; j >= 0; --j) {\n")],
    # gate applied at every sub-step instead of once per token
    "gate_every_substep": [(GATE, ""),
                           ("            const double bb = (double)J->beta[row];\n",
                            "            const double bb = (double)J->beta[row];\n"
                            "            if (J->g) { const double gt = (double)J->g[(b * T + t) * H + h];"
                            " for (int64_t i = 0; i < dk * dv; ++i) S[i] *= gt; }\n")],
    # gate applied after the sub-steps (also decays the token's own writes)
    "gate_after_substeps": [(GATE, ""),
                            (READOUT, GATE + READOUT)],
    # the key of sub-step 0 reused for every sub-step
    "wrong_substep_key": [("const float *kk = J->k + row * dk;",
                           "const float *kk = J->k + (((b * T + t) * n_h + 0) * H + h) * dk;")],
    # the initial state ignored
    "h0_ignored": [("    if (J->h0) {\n        const float *src",
                    "    if (0) {\n        const float *src")],
    # the readout uses the gate-free previous state's transpose orientation
    # (o = S q instead of S^T q) -- only well-defined for square states, so the
    # edit swaps the roles of the two loops' indices when dk == dv and is a
    # no-op otherwise
    "readout_transposed": [("acc += S[d * dv + c] * (double)qq[d];",
                            "acc += (dk == dv ? S[c * dv + d] : S[d * dv + c]) * (double)qq[d];")],
}


def _fix_readout_before(src):
    # remove the original readout (after the sub-steps) once the copy has been
    # placed before them
    first = src.find(READOUT)
    second = src.find(READOUT, first + len(READOUT))
    assert first >= 0 and second > first
    return src[:second] + src[second + len(READOUT):]


@functools.lru_cache(maxsize=None)
def _build(name, tmpdir):
    src = open(SRC, encoding="utf-8").read()
    for old, new in MUTANTS[name]:
        assert old in src, (name, old)
        src = src.replace(old, new, 1)
    if name == "readout_before_update":
        src = _fix_readout_before(src)
    cpath = os.path.join(tmpdir, f"{name}.c")
    lpath = os.path.join(tmpdir, f"lib{name}.so")
    with open(cpath, "w", encoding="utf-8") as f:
        f.write(src)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread",
                    "-o", lpath, cpath], check=True)
    return lpath


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path_factory):
    tmpdir = str(tmp_path_factory.getbasetemp())
    lib = oracle.load_library(_build(name, tmpdir))
    fwd = functools.partial(oracle.fwd, lib=lib)
    failed = []
    for check in ALL_CHECKS:
        try:
            check(fwd, np.random.default_rng(20261202))
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"no pin catches the planted mistake '{name}'"


def test_unmutated_copy_passes(tmp_path):
    """Control: the same build route with no edit passes every pin."""
    src = open(SRC, encoding="utf-8").read()
    cpath = tmp_path / "same.c"
    cpath.write_text(src, encoding="utf-8")
    lpath = str(tmp_path / "libsame.so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread",
                    "-o", lpath, str(cpath)], check=True)
    fwd = functools.partial(oracle.fwd, lib=oracle.load_library(lpath))
    for check in ALL_CHECKS:
        check(fwd, np.random.default_rng(20261202))


# --- the comparison metric and the decode entry point -----------------------
def _rel_squared(x, ref):
    x, ref = np.asarray(x, float), np.asarray(ref, float)
    den = np.sum(ref * ref)
    return float(np.sum((x - ref) ** 2) / den) if den else float(np.sum((x - ref) ** 2))


def _rel_unnormalised(x, ref):
    return float(np.linalg.norm((np.asarray(x, float) - np.asarray(ref, float)).ravel()))


def _rel_swapped(x, ref):
    return oracle.rel_l2(ref, x)


def _rel_maxabs(x, ref):
    x, ref = np.asarray(x, float), np.asarray(ref, float)
    den = np.abs(ref).max()
    return float(np.abs(x - ref).max() / den) if den else float(np.abs(x - ref).max())


def _rel_per_row_mean(x, ref):
    x, ref = np.atleast_2d(np.asarray(x, float)), np.atleast_2d(np.asarray(ref, float))
    rows = [oracle.rel_l2(a, b) for a, b in zip(x.reshape(x.shape[0], -1),
                                                 ref.reshape(ref.shape[0], -1))]
    return float(np.mean(rows))


REL_MUTANTS = {"squared_norms": _rel_squared, "unnormalised": _rel_unnormalised,
               "arguments_swapped": _rel_swapped, "max_abs": _rel_maxabs,
               "per_row_mean": _rel_per_row_mean}


@pytest.mark.parametrize("name", sorted(REL_MUTANTS))
def test_rel_l2_mutant_is_caught(name):
    from pins import check_rel_l2
    with pytest.raises(AssertionError):
        check_rel_l2(REL_MUTANTS[name])


def _step_state_f32(q, k, v, beta, g, state, *, n_h=1, **kw):
    # the carried state rounded to float32 before every call
    st = None if state is None else np.asarray(state, np.float32).astype(np.float64)
    return oracle.step(q, k, v, beta, g, st, n_h=n_h, **kw)


def _step_no_gate(q, k, v, beta, g, state, *, n_h=1, **kw):
    return oracle.step(q, k, v, beta, None, state, n_h=n_h, **kw)


def _step_no_carry(q, k, v, beta, g, state, *, n_h=1, **kw):
    return oracle.step(q, k, v, beta, g, None, n_h=n_h, **kw)


def _step_last_substep_only(q, k, v, beta, g, state, *, n_h=1, **kw):
    k, v, beta = np.asarray(k), np.asarray(v), np.asarray(beta)
    return oracle.step(q, k[:, -1:], v[:, -1:], beta[:, -1:], g, state, n_h=1, **kw)


STEP_MUTANTS = {"state_rounded_to_f32": _step_state_f32, "gate_dropped": _step_no_gate,
                "state_not_carried": _step_no_carry,
                "last_substep_only": _step_last_substep_only}


@pytest.mark.parametrize("name", sorted(STEP_MUTANTS))
def test_step_mutant_is_caught(name):
    from pins import check_step_chain, check_step_recall
    bad = STEP_MUTANTS[name]
    caught = []
    for check in (lambda: check_step_recall(bad, np.random.default_rng(20261203)),
                  lambda: check_step_chain(bad, oracle.fwd, np.random.default_rng(20261204))):
        try:
            check()
        except AssertionError:
            caught.append(True)
    assert caught, f"no pin catches the planted mistake '{name}' in the decode step"
