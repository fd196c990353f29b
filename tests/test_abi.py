"""The C-ABI library on a machine without a GPU: it loads, exports every
symbol include/delta.h declares, and rejects bad arguments before touching
CUDA (no compute call is made here)."""
import ctypes
import os
import re

import pytest

import weight_rnn_gb300 as wr
from weight_rnn_gb300 import build as wbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "delta.h")


@pytest.fixture(scope="module")
def lib():
    wbuild.build()
    return wr.load_library()


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(delta_[a-z_]+)\s*\(", text)))


def test_header_declarations_match_binding():
    assert declared_functions() == sorted(wr.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_library_has_no_cudart_runtime_dependency():
    # the CUDA runtime is linked statically so the library loads without a GPU
    with open(wr.library_path(), "rb") as f:
        data = f.read()
    assert b"libcudart.so" not in data


def test_status_strings(lib):
    assert wr.delta_status_string(wr.DELTA_OK) == "success"
    for st in (wr.DELTA_ERR_INVALID, wr.DELTA_ERR_UNSUPPORTED, wr.DELTA_ERR_ALIGN,
               wr.DELTA_ERR_CUDA):
        assert wr.delta_status_string(st) not in ("success", "unknown status")
    assert wr.delta_status_string(12345) == "unknown status"
    assert wr.delta_version() >= 100


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails first


def fwd(lib, **kw):
    a = dict(q=FAKE, k=FAKE * 2, v=FAKE * 3, beta=FAKE * 4, g=None, h0=None,
             out=FAKE * 5, hT=None, B=1, H=1, T=4, dk=16, dv=16, n_h=1, chunk=16,
             dtype=wr.DELTA_F32)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.delta_fwd(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["beta"]), vp(a["g"]),
                         vp(a["h0"]), vp(a["out"]), vp(a["hT"]), a["B"], a["H"], a["T"],
                         a["dk"], a["dv"], a["n_h"], a["chunk"], a["dtype"], None)


def step(lib, **kw):
    a = dict(q=FAKE, k=FAKE * 2, v=FAKE * 3, beta=FAKE * 4, g=None, state=FAKE * 5,
             out=FAKE * 6, B=1, H=1, dk=16, dv=16, n_h=1, dtype=wr.DELTA_F32)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.delta_step(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["beta"]), vp(a["g"]),
                          vp(a["state"]), vp(a["out"]), a["B"], a["H"], a["dk"], a["dv"],
                          a["n_h"], a["dtype"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(dk=48), wr.DELTA_ERR_UNSUPPORTED),
    (dict(dv=256), wr.DELTA_ERR_UNSUPPORTED),
    (dict(chunk=128), wr.DELTA_ERR_UNSUPPORTED),
    (dict(chunk=8), wr.DELTA_ERR_UNSUPPORTED),
    (dict(n_h=0), wr.DELTA_ERR_UNSUPPORTED),
    (dict(n_h=5), wr.DELTA_ERR_UNSUPPORTED),
    (dict(B=-1), wr.DELTA_ERR_INVALID),
    (dict(T=-3), wr.DELTA_ERR_INVALID),
    (dict(dtype=7), wr.DELTA_ERR_INVALID),
    (dict(q=None), wr.DELTA_ERR_INVALID),
    (dict(beta=None), wr.DELTA_ERR_INVALID),
    (dict(out=None), wr.DELTA_ERR_INVALID),
    (dict(k=FAKE + 8), wr.DELTA_ERR_ALIGN),
    (dict(hT=FAKE * 7 + 4), wr.DELTA_ERR_ALIGN),
    (dict(out=FAKE + 16), wr.DELTA_ERR_INVALID),         # out overlaps q
    (dict(hT=FAKE * 3), wr.DELTA_ERR_INVALID),           # hT overlaps v
    (dict(h0=FAKE * 8, hT=FAKE * 8 + 16), wr.DELTA_ERR_INVALID),  # partial overlap
    (dict(B=1 << 16, H=1 << 15), wr.DELTA_ERR_UNSUPPORTED),
])
def test_fwd_rejects_before_launch(lib, kw, status):
    assert fwd(lib, **kw) == status
    assert wr.delta_last_error() != ""


def test_fwd_empty_batch_is_ok_without_gpu(lib):
    # B*H == 0 is a valid empty problem: nothing is enqueued
    assert fwd(lib, B=0) == wr.DELTA_OK
    assert fwd(lib, H=0, q=None, k=None, v=None, beta=None, out=None) == wr.DELTA_OK


@pytest.mark.parametrize("kw,status", [
    (dict(dk=8), wr.DELTA_ERR_UNSUPPORTED),
    (dict(n_h=9), wr.DELTA_ERR_UNSUPPORTED),
    (dict(H=-2), wr.DELTA_ERR_INVALID),
    (dict(state=None), wr.DELTA_ERR_INVALID),
    (dict(g=FAKE * 9 + 2), wr.DELTA_ERR_ALIGN),
    (dict(out=FAKE + 32), wr.DELTA_ERR_INVALID),
    (dict(state=FAKE * 2), wr.DELTA_ERR_INVALID),
])
def test_step_rejects_before_launch(lib, kw, status):
    assert step(lib, **kw) == status


def test_binding_refuses_cpu_tensors(lib):
    import torch
    q = torch.zeros(1, 4, 1, 16)
    with pytest.raises(ValueError):
        wr.delta_fwd(q, q, torch.zeros(1, 4, 1, 16), torch.zeros(1, 4, 1))


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(wr, "_lib", None)
    monkeypatch.setattr(wr, "library_path", lambda: str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="missing"):
        wr.load_library()


def test_injected_failure_returns_before_launch(lib):
    """The host-side failure hook: after validation, before any CUDA call
    (the fake pointers are never touched), the caller sees DELTA_ERR_CUDA."""
    try:
        assert lib.delta_inject_failure(-1) == wr.DELTA_ERR_INVALID
        assert lib.delta_inject_failure(2) == wr.DELTA_OK
        assert fwd(lib) == wr.DELTA_ERR_CUDA
        assert "injected" in wr.delta_last_error()
        assert step(lib) == wr.DELTA_ERR_CUDA
        assert "injected" in wr.delta_last_error()
        # validation comes first and does not use up an injection
        assert lib.delta_inject_failure(1) == wr.DELTA_OK
        assert fwd(lib, dk=48) == wr.DELTA_ERR_UNSUPPORTED
        assert fwd(lib) == wr.DELTA_ERR_CUDA
    finally:
        lib.delta_inject_failure(0)


def test_selftest_wait_rejects_bad_poll_counts(lib):
    assert lib.delta_selftest_wait(0, None) == wr.DELTA_ERR_INVALID
    assert lib.delta_selftest_wait((1 << 24) + 1, None) == wr.DELTA_ERR_INVALID


def ut(lib, **kw):
    a = dict(k=FAKE * 2, beta=FAKE * 4, g=None, t=FAKE * 64, B=1, H=1, T=4, dk=128, n_h=1,
             chunk=64, dtype=wr.DELTA_BF16)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.delta_ut_transform(vp(a["k"]), vp(a["beta"]), vp(a["g"]), vp(a["t"]), a["B"],
                                  a["H"], a["T"], a["dk"], a["n_h"], a["chunk"], a["dtype"], None)


def fwd_ut(lib, **kw):
    a = dict(q=FAKE, k=FAKE * 2, v=FAKE * 3, beta=FAKE * 4, g=None, h0=None, t=FAKE * 64,
             out=FAKE * 5, hT=None, B=1, H=1, T=4, dk=128, dv=128, n_h=1, chunk=64,
             dtype=wr.DELTA_BF16)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.delta_fwd_with_ut(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["beta"]), vp(a["g"]),
                                 vp(a["h0"]), vp(a["t"]), vp(a["out"]), vp(a["hT"]), a["B"],
                                 a["H"], a["T"], a["dk"], a["dv"], a["n_h"], a["chunk"],
                                 a["dtype"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(dk=64), wr.DELTA_ERR_UNSUPPORTED),           # the UT pass is the tensor-core shape only
    (dict(chunk=32), wr.DELTA_ERR_UNSUPPORTED),
    (dict(dtype=wr.DELTA_F32), wr.DELTA_ERR_UNSUPPORTED),
    (dict(dtype=9), wr.DELTA_ERR_INVALID),
    (dict(n_h=5), wr.DELTA_ERR_UNSUPPORTED),
    (dict(T=-1), wr.DELTA_ERR_INVALID),
    (dict(k=None), wr.DELTA_ERR_INVALID),
    (dict(t=None), wr.DELTA_ERR_INVALID),
    (dict(t=FAKE * 64 + 8), wr.DELTA_ERR_ALIGN),
    (dict(t=FAKE * 2 + 16), wr.DELTA_ERR_INVALID),      # t_mat overlaps k
])
def test_ut_transform_rejects_before_launch(lib, kw, status):
    assert ut(lib, **kw) == status


def test_ut_transform_empty_is_ok_without_gpu(lib):
    assert ut(lib, B=0) == wr.DELTA_OK
    assert ut(lib, T=0, k=None, t=None) == wr.DELTA_OK


@pytest.mark.parametrize("kw,status", [
    (dict(dk=64, dv=64), wr.DELTA_ERR_UNSUPPORTED),
    (dict(dtype=wr.DELTA_F32), wr.DELTA_ERR_UNSUPPORTED),
    (dict(t=None), wr.DELTA_ERR_INVALID),
    (dict(t=FAKE * 5), wr.DELTA_ERR_INVALID),           # t_mat overlaps out
    (dict(t=FAKE * 64 + 4), wr.DELTA_ERR_ALIGN),
    (dict(q=None), wr.DELTA_ERR_INVALID),
])
def test_fwd_with_ut_rejects_before_launch(lib, kw, status):
    assert fwd_ut(lib, **kw) == status


def test_kernel_count(lib):
    assert lib.delta_fwd_kernel_count(4, 32, 8192, 128, 128, 1, 64, wr.DELTA_BF16) == 2
    assert lib.delta_fwd_kernel_count(1, 1, 64, 16, 16, 1, 16, wr.DELTA_F32) == 1
    assert lib.delta_fwd_kernel_count(0, 1, 64, 128, 128, 1, 64, wr.DELTA_BF16) == 0
    assert lib.delta_fwd_kernel_count(1, 1, 64, 48, 16, 1, 16, wr.DELTA_F32) == -1


def test_erank_rejects_bad_arguments(lib):
    P = [ctypes.c_void_p((i + 1) << 40) for i in range(2)]
    assert lib.delta_state_erank(P[0], P[1], -1, 1, 128, 128, None) == wr.DELTA_ERR_INVALID
    assert lib.delta_state_erank(P[0], P[1], 1, 1, 96, 128, None) == wr.DELTA_ERR_UNSUPPORTED
    assert lib.delta_state_erank(None, P[1], 1, 1, 128, 128, None) == wr.DELTA_ERR_INVALID
    assert lib.delta_state_erank(ctypes.c_void_p((1 << 40) + 8), P[1], 1, 1, 128, 128, None) == wr.DELTA_ERR_ALIGN
    # erank inside the state
    assert lib.delta_state_erank(P[0], ctypes.c_void_p((1 << 40) + 1024), 1, 1, 128, 128, None) == wr.DELTA_ERR_INVALID
    assert lib.delta_state_erank(P[0], P[1], 0, 5, 128, 128, None) == wr.DELTA_OK


def test_attention_map_rejects_bad_arguments(lib):
    P = [ctypes.c_void_p((i + 1) << 40) for i in range(5)]
    call = lambda *a: lib.delta_attention_map(*a)
    assert call(P[0], P[1], P[2], None, P[4], 1, 1, 65, 128, wr.DELTA_BF16, None) == wr.DELTA_ERR_UNSUPPORTED
    assert call(P[0], P[1], P[2], None, P[4], 1, 1, 64, 96, wr.DELTA_BF16, None) == wr.DELTA_ERR_UNSUPPORTED
    assert call(P[0], P[1], P[2], None, P[4], 1, 1, 8, 128, 7, None) == wr.DELTA_ERR_INVALID
    assert call(None, P[1], P[2], None, P[4], 1, 1, 8, 128, wr.DELTA_BF16, None) == wr.DELTA_ERR_INVALID
    assert call(P[0], P[1], P[2], None, P[0], 1, 1, 8, 128, wr.DELTA_BF16, None) == wr.DELTA_ERR_INVALID
    assert call(P[0], P[1], P[2], None, P[4], 1, 1, 0, 128, wr.DELTA_BF16, None) == wr.DELTA_OK


def fwd_prologue(lib, beta_map=0, **kw):
    a = dict(q=FAKE, k=FAKE * 2, v=FAKE * 3, beta=FAKE * 4, g=None, h0=None,
             out=FAKE * 5, hT=None, B=1, H=1, T=4, dk=16, dv=16, n_h=1, chunk=16,
             dtype=wr.DELTA_F32)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.delta_fwd_prologue(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["beta"]), vp(a["g"]),
                                  vp(a["h0"]), vp(a["out"]), vp(a["hT"]), a["B"], a["H"], a["T"],
                                  a["dk"], a["dv"], a["n_h"], a["chunk"], a["dtype"], beta_map,
                                  None)


def step_prologue(lib, beta_map=0, **kw):
    a = dict(q=FAKE, k=FAKE * 2, v=FAKE * 3, beta=FAKE * 4, g=None, state=FAKE * 5,
             out=FAKE * 6, B=1, H=1, dk=16, dv=16, n_h=1, dtype=wr.DELTA_F32)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.delta_step_prologue(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["beta"]),
                                   vp(a["g"]), vp(a["state"]), vp(a["out"]), a["B"], a["H"],
                                   a["dk"], a["dv"], a["n_h"], a["dtype"], beta_map, None)


@pytest.mark.parametrize("beta_map,kw,status", [
    (2, {}, wr.DELTA_ERR_INVALID),                       # unknown beta map
    (-1, {}, wr.DELTA_ERR_INVALID),
    (0, dict(dk=48), wr.DELTA_ERR_UNSUPPORTED),
    (1, dict(k=FAKE + 8), wr.DELTA_ERR_ALIGN),
    (1, dict(out=FAKE + 16), wr.DELTA_ERR_INVALID),      # out overlaps q_raw
    (0, dict(beta=None), wr.DELTA_ERR_INVALID),
])
def test_prologue_entry_points_reject_before_launch(lib, beta_map, kw, status):
    assert fwd_prologue(lib, beta_map, **kw) == status
    step_kw = {k: v for k, v in kw.items() if k in ("dk", "k", "beta")}
    if "out" in kw:
        step_kw["out"] = FAKE + 32
    assert step_prologue(lib, beta_map, **step_kw) == status


def test_prologue_empty_problems_are_ok_without_gpu(lib):
    assert fwd_prologue(lib, 1, B=0) == wr.DELTA_OK
    assert step_prologue(lib, 1, H=0) == wr.DELTA_OK


def test_binding_rejects_unknown_beta_map():
    import torch
    q = torch.zeros(1, 4, 1, 16)
    with pytest.raises(ValueError):
        wr.delta_fwd_prologue(q, q, q, torch.zeros(1, 4, 1), beta_map="tanh")
    with pytest.raises(ValueError):
        wr.delta_step_prologue(q[:, 0], q[:, :1], q[:, :1], torch.zeros(1, 1, 1), None,
                               torch.zeros(1, 1, 16, 16), beta_map="relu")


def prologue(lib, beta_map=0, **kw):
    a = dict(q=FAKE, k=FAKE * 2, beta=FAKE * 3, qo=FAKE * 4, ko=FAKE * 5, bo=FAKE * 6,
             B=1, H=1, T=4, dk=16, n_h=1, dtype=wr.DELTA_F32)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.delta_prologue(vp(a["q"]), vp(a["k"]), vp(a["beta"]), vp(a["qo"]), vp(a["ko"]),
                              vp(a["bo"]), a["B"], a["H"], a["T"], a["dk"], a["n_h"], a["dtype"],
                              beta_map, None)


@pytest.mark.parametrize("beta_map,kw,status", [
    (5, {}, wr.DELTA_ERR_INVALID),
    (0, dict(dk=24), wr.DELTA_ERR_UNSUPPORTED),
    (0, dict(n_h=0), wr.DELTA_ERR_UNSUPPORTED),
    (1, dict(T=-1), wr.DELTA_ERR_INVALID),
    (1, dict(dtype=3), wr.DELTA_ERR_INVALID),
    (0, dict(ko=None), wr.DELTA_ERR_INVALID),
    (0, dict(bo=FAKE * 6 + 4), wr.DELTA_ERR_ALIGN),
    (0, dict(qo=FAKE * 2 + 32), wr.DELTA_ERR_INVALID),   # q_out overlaps k_raw
    (1, dict(ko=FAKE * 4 + 16), wr.DELTA_ERR_INVALID),   # k_out overlaps q_out
])
def test_prologue_rejects_before_launch(lib, beta_map, kw, status):
    assert prologue(lib, beta_map, **kw) == status


def test_prologue_empty_is_ok_without_gpu(lib):
    assert prologue(lib, 0, T=0) == wr.DELTA_OK
    assert prologue(lib, 1, B=0, q=None, k=None) == wr.DELTA_OK


def fwd_kda(lib, **kw):
    a = dict(q=FAKE, k=FAKE * 2, v=FAKE * 3, beta=FAKE * 4, alpha=FAKE * 9, h0=None,
             out=FAKE * 5, hT=None, B=1, H=1, T=4, dk=16, dv=16, n_h=1, chunk=16,
             dtype=wr.DELTA_F32)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.delta_fwd_kda(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["beta"]), vp(a["alpha"]),
                             vp(a["h0"]), vp(a["out"]), vp(a["hT"]), a["B"], a["H"], a["T"],
                             a["dk"], a["dv"], a["n_h"], a["chunk"], a["dtype"], None)


def step_kda(lib, **kw):
    a = dict(q=FAKE, k=FAKE * 2, v=FAKE * 3, beta=FAKE * 4, alpha=FAKE * 9, state=FAKE * 5,
             out=FAKE * 6, B=1, H=1, dk=16, dv=16, n_h=1, dtype=wr.DELTA_F32)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.delta_step_kda(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["beta"]), vp(a["alpha"]),
                              vp(a["state"]), vp(a["out"]), a["B"], a["H"], a["dk"], a["dv"],
                              a["n_h"], a["dtype"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(alpha=None), wr.DELTA_ERR_INVALID),
    (dict(alpha=FAKE * 9 + 4), wr.DELTA_ERR_ALIGN),
    (dict(out=FAKE * 9 + 16), wr.DELTA_ERR_INVALID),     # out overlaps alpha
    (dict(dk=24), wr.DELTA_ERR_UNSUPPORTED),
    (dict(q=None), wr.DELTA_ERR_INVALID),
])
def test_kda_entry_points_reject_before_launch(lib, kw, status):
    assert fwd_kda(lib, **kw) == status
    skw = dict(kw)
    if "out" in skw:
        skw = dict(state=FAKE * 9 + 16)                  # state overlaps alpha
    assert step_kda(lib, **skw) == status


def test_kda_empty_problems_are_ok_without_gpu(lib):
    assert fwd_kda(lib, B=0) == wr.DELTA_OK
    assert step_kda(lib, H=0) == wr.DELTA_OK


def bwd(lib, **kw):
    a = dict(q=FAKE, k=FAKE * 2, v=FAKE * 3, beta=FAKE * 4, g=None, h0=None, dout=FAKE * 5,
             dhT=None, gq=FAKE * 6, gk=FAKE * 7, gv=FAKE * 8, gb=FAKE * 9, gg=None, gh0=None,
             B=1, H=1, T=4, dk=16, dv=16, n_h=1, dtype=wr.DELTA_F32)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.delta_bwd(*(vp(a[n]) for n in ("q", "k", "v", "beta", "g", "h0", "dout", "dhT",
                                             "gq", "gk", "gv", "gb", "gg", "gh0")),
                         a["B"], a["H"], a["T"], a["dk"], a["dv"], a["n_h"], a["dtype"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(dk=48), wr.DELTA_ERR_UNSUPPORTED),
    (dict(n_h=5), wr.DELTA_ERR_UNSUPPORTED),
    (dict(T=-1), wr.DELTA_ERR_INVALID),
    (dict(dtype=9), wr.DELTA_ERR_INVALID),
    (dict(dout=None), wr.DELTA_ERR_INVALID),
    (dict(gk=None), wr.DELTA_ERR_INVALID),
    (dict(g=FAKE * 10), wr.DELTA_ERR_INVALID),          # g given without its gradient
    (dict(gq=FAKE * 6 + 8), wr.DELTA_ERR_ALIGN),
    (dict(gq=FAKE * 5 + 16), wr.DELTA_ERR_INVALID),     # grad_q overlaps dout
    (dict(gv=FAKE * 7 + 16), wr.DELTA_ERR_INVALID),     # grad_v overlaps grad_k
])
def test_bwd_rejects_before_launch(lib, kw, status):
    assert bwd(lib, **kw) == status


def test_bwd_empty_batch_is_ok_without_gpu(lib):
    assert bwd(lib, B=0) == wr.DELTA_OK


def test_bwd_rejects_a_grid_too_large_for_its_column_groups(lib):
    # B*H = 2^30 passes the per-head limit, but four groups of 32 value
    # columns (dv = 128) would need 2^32 CTAs; the pointers are spaced far
    # enough apart that no range overlaps, and nothing is dereferenced
    span = 1 << 44
    kw = {n: span * (i + 1) for i, n in enumerate(("q", "k", "v", "beta", "dout", "gq", "gk",
                                                    "gv", "gb"))}
    assert bwd(lib, B=1 << 15, H=1 << 15, T=1, dk=16, dv=128, **kw) == wr.DELTA_ERR_UNSUPPORTED


def test_every_compute_binding_refuses_cpu_tensors(lib):
    # no CPU fallback anywhere: each compute call raises on host tensors
    # before reaching the library
    import torch
    B, T, H, d = 1, 4, 1, 16
    q, k, v = torch.zeros(B, T, H, d), torch.zeros(B, T, H, d), torch.zeros(B, T, H, d)
    beta, g = torch.zeros(B, T, H), torch.ones(B, T, H)
    state = torch.zeros(B, H, d, d)
    alpha_t, alpha_1 = torch.ones(B, T, H, d), torch.ones(B, H, d)
    q1, k1, b1, g1 = q[:, 0], k[:, :1], beta[:, :1], g[:, 0]
    calls = [
        lambda: wr.delta_fwd(q, k, v, beta, g),
        lambda: wr.delta_bwd(q, k, v, beta, g, state, v, state),
        lambda: wr.delta_fwd_kda(q, k, v, beta, alpha_t),
        lambda: wr.delta_step_kda(q1, k1, k1, b1, alpha_1, state),
        lambda: wr.delta_prologue(q, k, beta),
        lambda: wr.delta_fwd_prologue(q, k, v, beta, g),
        lambda: wr.delta_fwd_static_scratch(q, k, v, beta, g),
        lambda: wr.delta_state_erank(state),
        lambda: wr.delta_attention_map(q, k, beta, g),
        lambda: wr.delta_ut_transform(k, beta, g),
        lambda: wr.delta_fwd_with_ut(q, k, v, beta, g, None, torch.zeros(1, 64, 64)),
        lambda: wr.delta_step(q1, k1, k1, b1, g1, state),
        lambda: wr.delta_step_prologue(q1, k1, k1, b1, g1, state),
    ]
    for call in calls:
        with pytest.raises(ValueError, match="needs CUDA tensors"):
            call()
