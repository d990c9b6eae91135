"""GPU check of the tensor-core building blocks (TMA 128-byte-swizzled tile loads,
hand-swizzled tile writes, K-major and MN-major shared-memory descriptors, the instruction
descriptor, tcgen05.mma into TMEM and tcgen05.ld back) against a float64 matmul of the same
bf16 values.  Each case is one operand-layout combination that a library kernel uses."""
import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "tc_probe.cu")
LIB = os.path.join(HERE, "_build", "libtcprobe.so")


@pytest.fixture(scope="module")
def probe():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    hdr = os.path.join(ROOT, "efficient_transformer_gb300", "csrc", "la_tc_ptx.cuh")
    if not os.path.exists(LIB) or os.path.getmtime(LIB) < max(os.path.getmtime(SRC), os.path.getmtime(hdr)):
        subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                        "-Xcompiler", "-fPIC", "-shared", "-I", os.path.dirname(hdr), SRC, "-o", LIB],
                       check=True)
    lib = ctypes.CDLL(LIB)
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.tc_probe_mma.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, i, i, vp]
    lib.tc_probe_mma.restype = i
    return lib


CASES = [
    # N, K, a_mn, b_mn, a_manual, b_manual[, collector, dcol[, b_off]]   (M = 128)
    (32, 128, 0, 0, 0, 0),     # scores: phi(q) rows x phi(k) rows, 32 keys
    (128, 128, 0, 0, 0, 0),    # scores, 128 keys
    (64, 128, 0, 0, 0, 0),
    (128, 32, 0, 1, 1, 0),     # P (hand-written, K = 32 keys) x V (MN-major)
    (128, 128, 0, 1, 0, 0),    # phi(q) x state (MN-major)
    (128, 32, 1, 1, 0, 0),     # phi(k)^T (MN-major A) x V: state update
    (128, 64, 1, 1, 0, 0),
    (32, 128, 1, 1, 0, 1),     # phi(q)^T x dP (hand-written MN-major B, 32 keys)
    (32, 128, 1, 0, 0, 0),     # R^T (MN-major A) x phi(k) (K-major B)
    (64, 64, 0, 1, 0, 0),      # head dimension 64
    (128, 128, 0, 0, 1, 1),    # both hand-written
    (32, 128, 0, 0, 0, 0, 0, 192),    # accumulator at a column offset (dA')
    (128, 128, 0, 0, 0, 0, 0, 224),   # X
    (16, 128, 1, 0, 0, 0, 0, 480),    # r
    (32, 128, 0, 0, 0, 0, 1, 0),      # A kept in the collector buffer for a second MMA
    (128, 128, 1, 1, 0, 0, 1, 128),   # MN-major A and B
    (128, 32, 1, 1, 0, 0, 1, 64),     # S and z share phi(K)^T
    (32, 128, 0, 0, 0, 0, 2, 160),    # A (N = 32) then den (N = 16) from one read of phi(Q)
    (128, 128, 1, 0, 0, 0, 2, 352),   # R (N = 128) then r (N = 16), K-major B
    (128, 128, 0, 1, 0, 0, 2, 224),   # X then a narrower product from one read of g
    (16, 128, 1, 1, 0, 1, 0, 0, 32),  # gd as a column of the dP tile (MN-major B mid-block)
    (32, 128, 1, 1, 0, 1, 2, 0, 32),  # the same after a wider product that filled the collector
    (16, 128, 1, 1, 0, 1, 0, 0, 16),
    (32, 128, 1, 1, 0, 1, 3, 0),      # dk^T, r and R from one read of phi_s (fill, use, lastuse)
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "N{}_K{}_amn{}_bmn{}_am{}_bm{}".format(*c[:6])
                         + ("_coll{}_dcol{}".format(*c[6:8]) if len(c) > 6 else "")
                         + ("_boff{}".format(c[8]) if len(c) > 8 else ""))
def test_mma_layout(probe, case):
    N, K, a_mn, b_mn, a_man, b_man = case[:6]
    collector, dcol = case[6:8] if len(case) > 6 else (0, 0)
    b_off = case[8] if len(case) > 8 else 0
    M = 128
    g = torch.Generator().manual_seed(N * 1000 + K + 7 * a_mn + 13 * b_mn)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)    # logical A (m, k)
    B_all = torch.randn(N + b_off, K, generator=g).to(torch.bfloat16)
    B = B_all[b_off:]                                        # logical B (n, k)
    a_store = (A.t() if a_mn else A).contiguous().cuda()
    b_store = (B_all.t() if b_mn else B).contiguous().cuda()
    nout = {0: N, 1: 2 * N, 2: N + 16, 3: N + 32}[collector]
    d = torch.full((M, nout), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = probe.tc_probe_mma(a_store.data_ptr(), b_store.data_ptr(), d.data_ptr(), N, K, a_mn, b_mn,
                            a_man, b_man, collector, dcol, b_off, err.data_ptr())
    assert rc == 0, f"probe returned {rc}"
    want = A.double() @ B.double().t()
    if collector == 1:
        want = torch.cat([want, want], dim=1)
    elif collector == 2:
        want = torch.cat([want, want[:, :16]], dim=1)
    elif collector == 3:
        want = torch.cat([want, want[:, :16], want[:, :16]], dim=1)
    got = d.cpu().double()
    assert torch.isfinite(got).all()
    rel = float((got - want).abs().max() / want.abs().max())
    assert rel < 1e-5, f"max rel err {rel:.3e}"
