"""Helpers shared by the GPU parity tests: building/loading the library, device copies and
the elementwise tolerance |gpu - oracle| <= atol + rtol * |oracle|."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O

ATOL = 1e-2
RTOL = 1e-2
# Sums over tokens in the storage-model check: the fraction of elements allowed past the bound.
# When the fp32 evaluation rounds one large operand (h of 8 to 16 has a bf16 ulp of 1/16) to
# its other bf16 neighbour, every sum that operand enters moves by |other operand| x that
# ulp, up to about 0.3, whatever the sum's own size: a column of dW_d, for example.
SUM_FLIP_FRAC = 1e-6


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


def assert_close(gpu, ref, name, atol=ATOL, rtol=RTOL, reduction=False, extra=None,
                 allow_frac=0.0):
    """|gpu - oracle| <= atol + rtol |oracle| elementwise.

    Against the oracle's bf16-storage model this is the consistency check of the kernels'
    arithmetic; parity with the plain definition is ``check_plain``.

    ``reduction=True`` marks sums over the token axis (weight and gate gradients): there one
    operand element that the fp32 GPU evaluation rounds to the neighbouring bf16 value
    (unavoidable: about 1 in 2000 elements of a bf16 activation) moves every sum it enters
    by |other operand| x one bf16 ulp, independent of the sum's own value. The absolute
    term is then taken relative to the tensor's RMS: atol * max(1, rms(oracle)).

    ``extra`` adds an elementwise term to the bound (e.g. one bf16 ulp of each bf16 summand
    of a sum over slots). ``allow_frac`` lets that fraction of the elements fall outside:
    with FP8 operands a bf16 neighbour of h can round to the next E4M3 code, which moves a
    whole output row by a code step."""
    g = h64(gpu) if not isinstance(gpu, np.ndarray) else gpu.astype(np.float64)
    r = np.asarray(ref, dtype=np.float64)
    if reduction and r.size:
        atol = atol * max(1.0, float(np.sqrt(np.mean(r * r))))
    assert g.shape == r.shape, f"{name}: shape {g.shape} vs {r.shape}"
    err = np.abs(g - r)
    bound = atol + rtol * np.abs(r) + (0.0 if extra is None else extra)
    bad = err > bound
    if reduction:
        allow_frac = max(allow_frac, SUM_FLIP_FRAC)
    if bad.sum() <= allow_frac * bad.size:
        return
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), r.shape)
        where = [tuple(int(v) for v in w) for w in np.argwhere(bad)[:8]]
        raise AssertionError(
            f"{name}: {int(bad.sum())} of {bad.size} elements outside {atol} + {rtol}|ref|; "
            f"worst at {i}: gpu {g[i]!r} oracle {r[i]!r}; max abs err {err.max():.3e}; "
            f"first outside at {where}")


# Literal-tolerance report against the plain definition: per case and tensor, how many
# elements fall outside |gpu - oracle| <= ATOL + RTOL |oracle| and by how much, beside the
# same figures for the oracle's own bf16-storage model. Printed at the end of the session
# (tests/conftest.py) and written as JSON to $MOE_PARITY_REPORT when that is set.
REPORT = {"plain": [], "near_ties": []}


def exceedances(got, want) -> dict:
    """Elements outside the literal tolerance: count, worst excess over the bound and the
    largest absolute error."""
    g = h64(got) if not isinstance(got, np.ndarray) else got.astype(np.float64)
    w = np.asarray(want, dtype=np.float64)
    assert g.shape == w.shape, f"shape {g.shape} vs {w.shape}"
    if w.size == 0:
        return {"size": 0, "exceed": 0, "worst_excess": 0.0, "max_err": 0.0}
    err = np.abs(g - w)
    over = err - (ATOL + RTOL * np.abs(w))
    return {"size": int(w.size), "exceed": int((over > 0).sum()),
            "worst_excess": float(over.max()), "max_err": float(err.max())}


def check_plain(case, name, gpu, plain, storage):
    """Parity with the plain definition at the literal tolerance.

    ``plain`` is the oracle's exact fp64 value and ``storage`` the oracle's value when the
    tensors the workloads store in bf16 are rounded to bf16 (``rnd=bf16_round``). Elements
    outside the tolerance are recorded, not hidden. Storing activations in bf16 alone moves
    sums over thousands of tokens past the tolerance's absolute term, so the check is that the
    GPU goes outside it no more often, and by no more, than bf16 storage itself does: its
    count at most 1.5x the storage model's plus a few elements of chance (a sum within an
    ulp of the bound falls either way), and its worst excess at most 1.5x the storage
    model's plus a quarter of the absolute term."""
    g = exceedances(gpu, plain)
    s = exceedances(storage, plain)
    REPORT["plain"].append({"case": case, "tensor": name, **g, "storage_exceed": s["exceed"],
                            "storage_worst_excess": s["worst_excess"]})
    allow = 1.5 * s["exceed"] + 3.0 * np.sqrt(s["exceed"]) + 1e-5 * g["size"] + 2
    assert g["exceed"] <= allow, (
        f"{case} {name}: {g['exceed']} of {g['size']} elements outside the literal tolerance "
        f"(bf16 storage alone: {s['exceed']}); worst excess {g['worst_excess']:.3e}")
    assert g["worst_excess"] <= 1.5 * max(s["worst_excess"], 0.0) + 0.25 * ATOL, (
        f"{case} {name}: worst excess {g['worst_excess']:.3e} over the literal tolerance "
        f"(bf16 storage alone: {s['worst_excess']:.3e})")
    return g


def record_near_ties(case, near, T):
    REPORT["near_ties"].append({"case": case, "near_ties": int(near), "tokens": int(T)})


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


def dx_summand_ulps(fwd, bwd):
    """Per element of the layer's input gradient: one bf16 ulp of each of its bf16 summands
    (the token's expert input-gradient rows and the shared expert's), by which a different
    but correct rounding of each summand moves the sum."""
    s2r = fwd["slot_to_row"]
    b = np.zeros_like(bwd["dx"])
    for i in range(s2r.shape[1]):
        b += ulp_bf16(bwd["dX_perm"][s2r[:, i]])
    if "dx_shared" in bwd:
        b += ulp_bf16(bwd["dx_shared"])
    return b


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
