"""The tensor-core building blocks (csrc/umma.cuh) on the GPU, in isolation.

A probe kernel (tests/cuda/umma_check.cu, test-only) issues one tcgen05.mma of
kind::f16 (bf16 x bf16 -> fp32) from K-major 128-byte-swizzled shared-memory
tiles and dumps every TMEM lane.  Checks: the instruction and shared-memory
descriptors give D = A B^T; for M = 128 row i sits in lane i; the lane layout of
M = 64 is recorded (rows 16w..16w+15 in lanes 32w..32w+15); MN-major (transposed)
storage of A and / or B gives the same product; the 16x32bx2 TMEM load hands the
upper half of a warp the first 16 lanes at a second column offset."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def probe():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    src = os.path.join(HERE, "cuda", "umma_check.cu")
    lib = os.path.join(HERE, "cuda", "libumma_check.so")
    subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2",
                           "-std=c++17", "-shared", "-Xcompiler", "-fPIC", "-cudart", "shared",
                           "-I", os.path.join(ROOT, "gated_deltanet_backward_gb300", "csrc"),
                           src, "-o", lib])
    L = ctypes.CDLL(lib)
    L.umma_check.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 5 + [ctypes.c_void_p]
    L.umma_check.restype = ctypes.c_int
    L.tmem_x2_check.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    L.tmem_x2_check.restype = ctypes.c_int
    return torch, L


def _run(probe, M, N, K, seed=0, a_mn=False, b_mn=False):
    torch, L = probe
    g = torch.Generator().manual_seed(seed)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, generator=g).to(torch.bfloat16)
    dA, dB = A.cuda(), B.cuda()
    out = torch.full((128, N), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = L.umma_check(dA.data_ptr(), dB.data_ptr(), out.data_ptr(), M, N, K, int(a_mn),
                      int(b_mn), st.data_ptr())
    assert rc == 0 and int(st.item()) == 0
    ref = (A.double() @ B.double().T).numpy()
    return out.cpu().double().numpy(), ref


@pytest.mark.parametrize("N,K", [(16, 16), (64, 64), (64, 128), (128, 128), (256, 64), (32, 96)])
def test_m128_is_row_per_lane(probe, N, K):
    got, ref = _run(probe, 128, N, K)
    err = np.abs(got - ref).max() / np.abs(ref).max()
    assert err < 1e-5, err


@pytest.mark.parametrize("N,K", [(64, 128), (128, 64)])
def test_m64_lane_layout(probe, N, K):
    got, ref = _run(probe, 64, N, K)
    lanes = np.array([32 * (i // 16) + (i % 16) for i in range(64)])
    err = np.abs(got[lanes] - ref).max() / np.abs(ref).max()
    assert err < 1e-5, err


@pytest.mark.parametrize("M,N,K,a_mn,b_mn", [
    (128, 64, 64, True, False),    # dO^T P^T: A read from the natural dO tile
    (128, 128, 128, False, True),  # [dO; dDelta] S^T: B read from the S^T tile
    (128, 128, 64, True, True),
    (64, 128, 128, True, False),
    (64, 64, 64, False, True),
])
def test_mn_major_operands(probe, M, N, K, a_mn, b_mn):
    got, ref = _run(probe, M, N, K, seed=3, a_mn=a_mn, b_mn=b_mn)
    lanes = (np.arange(128) if M == 128 else
             np.array([32 * (i // 16) + (i % 16) for i in range(64)]))
    err = np.abs(got[lanes] - ref).max() / np.abs(ref).max()
    assert err < 1e-5, err


def test_tmem_ld16_x2_lane_layout(probe):
    torch, L = probe
    out = torch.full((4, 32, 4, 16), float("nan"), device="cuda")
    st = torch.ones(1, dtype=torch.int32, device="cuda")
    assert L.tmem_x2_check(out.data_ptr(), st.data_ptr()) == 0 and int(st.item()) == 0
    got = out.cpu().numpy()
    w, t, piece, j = np.meshgrid(np.arange(4), np.arange(32), np.arange(4), np.arange(16),
                                 indexing="ij")
    lane = 32 * w + (t % 16)
    col = 16 * piece + j + 64 * (t // 16)
    assert np.array_equal(got, (lane * 1000 + col).astype(np.float32))
