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
