"""Device random numbers: the kernels' Philox4x32-10 (generic and row-specialised)
against CUDA's curand_Philox4x32_10 and the oracle, bit for bit; the single-precision
Gumbel against binary64; and the soundness of the log-free rejection test."""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def lib():
    src = os.path.join(HERE, "cuda", "rng_check.cu")
    out_dir = os.path.join(HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "librngcheck.so")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-shared",
                    "-Xcompiler", "-fPIC", "-cudart", "shared", "-I", os.path.join(HERE, "..", "include"),
                    src, "-o", so], check=True)
    L = ctypes.CDLL(so)
    P = ctypes.c_void_p
    L.rng_check_philox.argtypes = [ctypes.c_int, P, P, P, P, ctypes.c_uint32, ctypes.c_uint32, P]
    L.rng_check_gumbel.argtypes = [ctypes.c_int, P, P, P, P]
    L.rng_check_gumbel_fast.argtypes = [ctypes.c_int, P, P]
    L.rng_check_reject_fast.argtypes = [ctypes.c_int, P, P, ctypes.c_float, P]
    return L


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_philox_matches_curand_and_oracle(lib):
    rng = np.random.default_rng(0)
    n = 1 << 16
    ctr = rng.integers(0, 2**32, (4, n), dtype=np.uint64).astype(np.uint32)
    ctr[:, :4] = [[0, 0xFFFFFFFF, 0x243F6A88, 7]] * 4  # include the known-answer counters' words
    k0, k1 = 0xA4093822, 0x299F31D0
    dev = [torch.from_numpy(ctr[i].view(np.int32)).cuda() for i in range(4)]
    out = torch.zeros(12 * n, dtype=torch.int32, device="cuda")
    assert lib.rng_check_philox(n, *[_p(d) for d in dev], k0, k1, _p(out)) == 0
    o = out.cpu().numpy().view(np.uint32).reshape(n, 3, 4)
    assert (o[:, 0] == o[:, 2]).all(), "generic rounds differ from curand_Philox4x32_10"
    assert (o[:, 1] == o[:, 2]).all(), "row-specialised rounds differ from curand_Philox4x32_10"
    for i in range(0, n, 4099):
        ref = oracle.philox4x32_10(ctr[:, i], [k0, k1])
        assert list(ref) == list(o[i, 0])


def test_gumbel_single_precision_accuracy(lib):
    # every 2^8-th 24-bit uniform code plus the extreme tail on both sides
    b24 = np.concatenate([np.arange(0, 1 << 24, 256), np.arange(0, 4096), np.arange((1 << 24) - 4096, 1 << 24)])
    bits = (b24.astype(np.uint64) << 8).astype(np.uint32)
    n = len(bits)
    tb = torch.from_numpy(bits.view(np.int32)).cuda()
    t = torch.zeros(n, dtype=torch.float32, device="cuda")
    g = torch.zeros(n, dtype=torch.float32, device="cuda")
    rej = torch.zeros(n, dtype=torch.int32, device="cuda")
    assert lib.rng_check_gumbel(n, _p(tb), _p(t), _p(g), _p(rej)) == 0
    u = (b24.astype(np.float64) + 0.5) / 2**24
    exact = -np.log(-np.log1p(u - 1.0))
    err = np.abs(g.cpu().numpy().astype(np.float64) - exact)
    # absolute accuracy of the key z + g: far inside the 1e-5 boundary window
    assert err.max() < 2e-6, err.max()


def test_fast_gumbel_single_precision_accuracy(lib):
    # the survivors' Gumbel of the draft epilogue: every 2^8-th 24-bit code, both tails,
    # and the codes around the branch point u = 1/2
    b24 = np.concatenate([np.arange(0, 1 << 24, 256), np.arange(0, 4096), np.arange((1 << 24) - 4096, 1 << 24),
                          np.arange((1 << 23) - 2048, (1 << 23) + 2048)])
    bits = (b24.astype(np.uint64) << 8).astype(np.uint32) | np.uint32(0xA5)  # low bits must not matter
    n = len(bits)
    tb = torch.from_numpy(bits.view(np.int32)).cuda()
    g = torch.zeros(n, dtype=torch.float32, device="cuda")
    assert lib.rng_check_gumbel_fast(n, _p(tb), _p(g)) == 0
    u = (b24.astype(np.float64) + 0.5) / 2**24
    exact = -np.log(-np.log1p(u - 1.0))
    err = np.abs(g.cpu().numpy().astype(np.float64) - exact)
    assert err.max() < 2e-6, (err.max(), b24[np.argmax(err)])


def test_rejection_test_is_sound(lib):
    # gumbel_cannot_win(bits, t) must imply E = -ln u >= t, i.e. g <= -ln t (so that
    # z + g <= best whenever t >= e^{z - best}); up to the rounding of 1-u below 1/2
    rng = np.random.default_rng(1)
    n = 1 << 20
    bits = rng.integers(0, 2**32, n, dtype=np.uint64).astype(np.uint32)
    bits[: n // 4] |= 0xFFF00000  # many draws near u -> 1 (large Gumbels)
    lt = rng.uniform(-25, 3, n)
    t = np.exp(lt).astype(np.float32)
    tb = torch.from_numpy(bits.view(np.int32)).cuda()
    g = torch.zeros(n, dtype=torch.float32, device="cuda")
    rej = torch.zeros(n, dtype=torch.int32, device="cuda")
    assert lib.rng_check_gumbel(n, _p(tb), _p(torch.from_numpy(t).cuda()), _p(g), _p(rej)) == 0
    rej = rej.cpu().numpy().astype(bool)
    u = ((bits >> 8).astype(np.float64) + 0.5) / 2**24
    g64 = -np.log(-np.log1p(u - 1.0))
    assert (g64[rej] <= -np.log(t[rej].astype(np.float64)) + 1e-6).all()
    assert rej.mean() > 0.5  # and it does reject most draws


@pytest.mark.parametrize("scale", [1.0, 0.37, 3.0e4])
def test_conversion_free_rejection_is_sound(lib, scale):
    # the draft epilogue's form, fl(t * scale + f) <= 2 - 2^-22 with f from the word's top 23
    # bits, must imply E = -ln u >= 1 - u >= t * scale, i.e. g <= -ln(t * scale)
    rng = np.random.default_rng(2)
    n = 1 << 20
    bits = rng.integers(0, 2**32, n, dtype=np.uint64).astype(np.uint32)
    bits[: n // 4] |= 0xFFF00000  # many draws near u -> 1
    u = (2.0 * (bits >> 8).astype(np.float64) + 1.0) / 2.0**25
    # thresholds at random, and within a few 1e-7 of 1 - u
    tt = np.where(rng.random(n) < 0.5, np.exp(rng.uniform(-25, 1, n)), (1.0 - u) * (1 + rng.normal(0, 3e-7, n)))
    t = (tt / scale).astype(np.float32)
    tb = torch.from_numpy(bits.view(np.int32)).cuda()
    rej = torch.zeros(n, dtype=torch.int32, device="cuda")
    assert lib.rng_check_reject_fast(n, _p(tb), _p(torch.from_numpy(t).cuda()), scale, _p(rej)) == 0
    rej = rej.cpu().numpy().astype(bool)
    prod = t.astype(np.float64) * float(np.float32(scale))  # the kernel's operands are binary32
    assert (1.0 - u[rej] >= prod[rej]).all()
    # it rejects whatever lies clearly below the exact boundary
    far = (1.0 - u) - prod > 2.0**-20
    assert rej[far].all()
