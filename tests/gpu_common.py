"""Helpers shared by the GPU parity tests: building/loading the library, device copies and
the elementwise tolerance |gpu - oracle| <= atol + rtol * |oracle|."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O

ATOL = 1e-2
RTOL = 1e-2


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from pretraining_sigmoid_softmax_gb300 import build, _lib
    build.build_library()
    _lib.load()


def dev(t):
    return t.contiguous().cuda()


def h64(t):
    return O.to64(t)


def assert_close(gpu, ref, name, atol=ATOL, rtol=RTOL, reduction=False):
    """|gpu - oracle| <= atol + rtol |oracle| elementwise.

    ``reduction=True`` marks sums over the token axis (weight and gate gradients): there one
    operand element that the fp32 GPU evaluation rounds to the neighbouring bf16 value
    (unavoidable: about 1 in 2000 elements of a bf16 activation) moves every sum it enters
    by |other operand| x one bf16 ulp, independent of the sum's own value. The absolute
    term is then taken relative to the tensor's RMS: atol * max(1, rms(oracle))."""
    g = h64(gpu) if not isinstance(gpu, np.ndarray) else gpu.astype(np.float64)
    r = np.asarray(ref, dtype=np.float64)
    if reduction and r.size:
        atol = atol * max(1.0, float(np.sqrt(np.mean(r * r))))
    assert g.shape == r.shape, f"{name}: shape {g.shape} vs {r.shape}"
    err = np.abs(g - r)
    bad = err > atol + rtol * np.abs(r)
    if bad.any():
        i = np.unravel_index(np.argmax(err - (atol + rtol * np.abs(r))), r.shape)
        raise AssertionError(
            f"{name}: {int(bad.sum())} of {bad.size} elements outside {atol} + {rtol}|ref|; "
            f"worst at {i}: gpu {g[i]!r} oracle {r[i]!r}; max abs err {err.max():.3e}")


def ulp_bf16(v):
    _, e = np.frexp(np.abs(np.asarray(v, dtype=np.float64)))
    return np.ldexp(1.0, np.maximum(e, -125) - 8)


def assert_gemm_exact(gpu, A, B, name):
    """gpu == bf16(A @ B) up to half a bf16 ulp plus the fp32 accumulation error bound
    (K + 2) * 2^-24 * (|A| @ |B|): the tensor-core result of exact bf16 operands."""
    g = h64(gpu)
    ex = A @ B
    bound = 0.5 * ulp_bf16(ex) * 1.001 + (A.shape[1] + 2) * 2.0 ** -24 * (np.abs(A) @ np.abs(B))
    bad = np.abs(g - ex) > bound
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{name}: {int(bad.sum())} of {bad.size} elements outside the "
                             f"bf16/fp32 bound; e.g. {i}: gpu {g[i]!r} exact {ex[i]!r}")


def padded_offsets(counts, align=128):
    c = np.asarray(counts, dtype=np.int64)
    return np.concatenate([[0], np.cumsum((c + align - 1) // align * align)]).astype(np.int64)


def gpu_rows(offsets, row_offsets):
    """Map each unpadded expert-major row p to its row in the padded layout."""
    E = len(offsets) - 1
    out = np.empty(int(offsets[-1]), dtype=np.int64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        out[lo:hi] = row_offsets[e] + np.arange(hi - lo)
    return out


def randn_bf16(shape, gen, std=1.0):
    return (torch.randn(shape, generator=gen) * std).to(torch.bfloat16)
