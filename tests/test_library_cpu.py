"""The C-ABI library builds, loads and exports every symbol its header declares; the
host-only entry points and argument checks work without a GPU."""
import ctypes
import os
import re
import shutil

import pytest

from pretraining_sigmoid_softmax_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_gb300.h")

needs_nvcc = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not installed")


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build_library()
    return _lib.load()


def test_header_declares_the_layer_entry_points():
    names = header_functions()
    for must in ("moe_route", "moe_permute", "moe_expert_fwd", "moe_combine", "moe_bias_update",
                 "moe_expert_bwd", "moe_combine_bwd", "moe_route_bwd", "moe_permute_bwd"):
        assert must in names
    assert set(names) == set(_lib.PROTOTYPES), "binding prototypes differ from the header"


@needs_nvcc
def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


@needs_nvcc
def test_host_only_entry_points(lib):
    assert lib.moe_version() >= 100
    assert lib.moe_status_string(0) == b"ok"
    assert lib.moe_status_string(6) == b"bounded device wait ran out"
    # capacity of the padded layout: round_up(T*k + E*127, 128)
    assert lib.moe_padded_rows(512, 2, 8) == 2048
    assert lib.moe_padded_rows(65536, 8, 64) == 532480
    assert lib.moe_padded_rows(1, 1, 1) == 128
    assert lib.moe_workspace_bytes(65536, 4096, 64, 8) >= 32 * 64 * 4096 * 4
    assert lib.moe_workspace_bytes(0, 1, 1, 1) == 0


@needs_nvcc
def test_argument_checks_return_before_any_device_work(lib):
    # null pointers are rejected on the host
    rc = lib.moe_route(None, None, None, 16, 128, 8, 2, 0, 0.0, None, None, None, None, None,
                       None, None, 0, None)
    assert rc == 1
    rc = lib.moe_permute(None, None, 16, 128, 8, 2, None, None, None, None, None, None, None, None,
                         None, 0, None)
    assert rc == 1
    rc = lib.moe_expert_fwd(None, None, 1, 16, 128, 128, None, None, None, None, None, None, None,
                            None, None, 0, None)
    assert rc == 1
    rc = lib.moe_bias_update(None, 8, 16, 2, 0.001, None, None)
    assert rc == 1
    rc = lib.moe_permute_fp8(None, None, None, None, None, 16, 128, 8, 2, None, None, None)
    assert rc == 1
    lib.moe_check_bounded_wait.argtypes = [ctypes.c_uint64, ctypes.c_void_p]
    assert lib.moe_check_bounded_wait(0, None) == 1  # a zero limit is rejected
    assert lib.moe_check_bounded_wait(2_000_000_000, None) == 1  # so is one above a second
    code = ctypes.c_int(0)
    assert lib.moe_device_status(None, None, None) == 1


@needs_nvcc
def test_padded_capacity_holds_every_routing(lib):
    """moe_padded_rows bounds the padded layout (each expert's segment rounded up to 128
    rows) for any split of the T*k routed rows over E experts, including the worst split,
    where E - 1 experts hold one row each and waste 127 padding rows apiece."""
    import numpy as np
    rng = np.random.default_rng(0)

    def padded(counts):
        return int(sum(-(-int(c) // 128) * 128 for c in counts))

    for T, k, E in [(1, 1, 1), (7, 2, 4), (300, 3, 6), (4096, 8, 64), (65536, 8, 64), (1000, 32, 256)]:
        cap = lib.moe_padded_rows(T, k, E)
        assert cap % 128 == 0 and cap >= T * k
        for _ in range(50):
            assert padded(rng.multinomial(T * k, rng.dirichlet(np.ones(E) * 0.3))) <= cap
        if T * k >= E:
            worst = np.ones(E, dtype=np.int64)
            worst[0] = T * k - (E - 1)
            assert padded(worst) <= cap


@needs_nvcc
def test_workspace_grows_with_every_size(lib):
    lib.moe_workspace_bytes.restype = ctypes.c_size_t
    base = (4096, 1024, 32, 4)
    w0 = lib.moe_workspace_bytes(*base)
    assert w0 > 0
    for i, bigger in enumerate([8192, 2048, 64, 8]):
        args = list(base)
        args[i] = bigger
        assert lib.moe_workspace_bytes(*args) >= w0, args


@needs_nvcc
def test_degenerate_and_inconsistent_arguments_are_rejected_on_the_host(lib):
    """Empty sizes, an unknown router mode, a router mode without its outputs, misaligned
    pointers and a half-given gate-folding pair return MOE_ERR_INVALID_ARG (1) before any
    device work (these checks come before the device check, so they hold without a GPU)."""
    P = 4096  # a stand-in device address (never dereferenced on the host), 16-byte aligned
    bad = P + 2  # not 16-byte aligned
    ws = P
    route = lambda x, b, T, mode, logits, lse, z: lib.moe_route(
        x, P, b, T, 256, 8, 2, mode, 0.0, logits, P, P, P, lse, z, ws, 1 << 20, None)
    assert route(P, P, 0, 0, P, P, P) == 1          # T = 0
    assert route(P, P, 16, 7, P, P, P) == 1         # unknown mode
    assert route(P, None, 16, 0, P, P, P) == 1      # sigmoid mode needs the bias
    assert route(P, None, 16, 1, None, P, P) == 1   # softmax mode needs logits, lse, z-loss
    assert route(bad, P, 16, 0, P, P, P) == 1       # misaligned x
    assert lib.moe_permute(P, P, 0, 256, 8, 2, P, P, P, P, P, P, None, None, ws, 1 << 20, None) == 1
    assert lib.moe_permute(P, bad, 16, 256, 8, 2, P, P, P, P, P, P, None, None, ws, 1 << 20,
                           None) == 1
    assert lib.moe_permute(P, P, 16, 256, 8, 2, P, P, P, P, P, P, P, None, ws, 1 << 20,
                           None) == 1   # the row gates need both pointers
    assert lib.moe_combine(P, P, P, None, 0, 256, 2, P, None) == 1
    assert lib.moe_combine(bad, P, P, None, 16, 256, 2, P, None) == 1
    fwd = lambda rows, E, ro, X: lib.moe_expert_fwd(X, ro, E, rows, 256, 128, P, P, P, P, P, P,
                                                     P, None, ws, 1 << 20, None)
    assert fwd(0, 1, None, P) == 1                  # no rows
    assert fwd(16, 2, None, P) == 1                 # no layout for two experts
    assert fwd(16, 1, None, bad) == 1               # misaligned operand
    bwd = lambda rg, gp, parts=7, dl=None, wr=None, ro=None: lib.moe_expert_bwd(
        P, P, P, P, P, ro, 1, 16, 256, 128, P, P, P, P, P, P, P, P, P, rg, gp, parts, dl, wr, ws,
        1 << 20, None)
    assert bwd(P, None) == 1 and bwd(None, P) == 1  # row gates and gate partials come together
    assert bwd(None, None, parts=0) == 1 and bwd(None, None, parts=8) == 1  # unknown parts
    assert bwd(None, None, dl=P) == 1 and bwd(None, None, wr=P) == 1  # router term: both or neither
    assert bwd(None, None, dl=P, wr=P) == 1         # the router term needs the routed layout
    assert bwd(None, None, dl=P, wr=bad, ro=P) == 1  # misaligned router weight
    rbwd = lambda mode, extra, s2r, dl: lib.moe_route_bwd(P, P, P, P, P, P, P, extra, 16, 256, 8,
                                                          2, mode, 0.0, P, P, s2r, dl, ws, 1 << 20,
                                                          None)
    assert rbwd(0, None, P, None) == 1 and rbwd(0, None, None, P) == 1  # rows: both or neither
    assert rbwd(1, None, P, P) == 1                 # softmax: the logit gradient is dense
    assert rbwd(0, P, P, P) == 1                    # an extra (dense) logit gradient
