"""Thin Python binding of the C ABI: one function per entry point, same names, arguments
are torch tensors (device memory) that are turned into raw pointers and sizes. No step of
the layer is computed here."""
from __future__ import annotations

import ctypes

import torch

from . import _lib

MODE_SIGMOID = 0
MODE_SOFTMAX = 1
ROW_ALIGN = 128


class MoEError(RuntimeError):
    pass


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, name: str):
    if rc != 0:
        msg = _lib.load().moe_status_string(rc).decode()
        raise MoEError(f"{name} failed: {msg} (status {rc})")


def _contig(*ts):
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise MoEError("tensors passed to the MoE library must be contiguous")


def status_string(rc: int) -> str:
    return _lib.load().moe_status_string(rc).decode()


def moe_version() -> int:
    return _lib.load().moe_version()


def moe_padded_rows(T: int, k: int, E: int) -> int:
    return _lib.load().moe_padded_rows(T, k, E)


def moe_workspace_bytes(T: int, d: int, E: int, k: int) -> int:
    return _lib.load().moe_workspace_bytes(T, d, E, k)


def moe_device_status(stream=None) -> tuple[int, int]:
    code, site = ctypes.c_int(0), ctypes.c_int(0)
    _check(_lib.load().moe_device_status(_stream(stream), ctypes.byref(code), ctypes.byref(site)),
           "moe_device_status")
    return code.value, site.value


def moe_clear_device_status(stream=None):
    _check(_lib.load().moe_clear_device_status(_stream(stream)), "moe_clear_device_status")


def moe_set_wait_limit_ns(ns: int):
    _lib.load().moe_set_wait_limit_ns(int(ns))


def moe_check_bounded_wait(limit_ns: int, stream=None):
    """One bounded wait that cannot complete: records MOE_ERR_TIMEOUT (site 90) and returns."""
    _check(_lib.load().moe_check_bounded_wait(int(limit_ns), _stream(stream)),
           "moe_check_bounded_wait")


def moe_route(x, W_r, b, k, mode, z_coef, logits, topk_idx, topk_gate, topk_score, lse, z_loss,
              ws, stream=None):
    T, d = x.shape
    E = W_r.shape[0]
    _contig(x, W_r, b, logits, topk_idx, topk_gate, topk_score, lse, z_loss, ws)
    _check(_lib.load().moe_route(_p(x), _p(W_r), _p(b), T, d, E, k, mode, float(z_coef),
                                 _p(logits), _p(topk_idx), _p(topk_gate), _p(topk_score), _p(lse),
                                 _p(z_loss), _p(ws), ws.numel(), _stream(stream)), "moe_route")


def moe_permute(topk_idx, x, E, counts, offsets, row_offsets, perm_token, slot_to_row, X_perm,
                ws, stream=None, topk_gate=None, row_gate=None):
    T, k = topk_idx.shape
    d = x.shape[1]
    _contig(topk_idx, x, counts, offsets, row_offsets, perm_token, slot_to_row, X_perm, ws)
    if row_gate is not None:
        _contig(topk_gate, row_gate)
    _check(_lib.load().moe_permute(_p(topk_idx), _p(x), T, d, E, k, _p(counts), _p(offsets),
                                   _p(row_offsets), _p(perm_token), _p(slot_to_row), _p(X_perm),
                                   _p(topk_gate), _p(row_gate), _p(ws), ws.numel(),
                                   _stream(stream)), "moe_permute")


def moe_permute_noalloc(topk_idx, x, E, counts, offsets, row_offsets, perm_token, slot_to_row,
                        X_perm, stream=None):
    """moe_permute without a workspace argument: its scratch is a fixed, library-owned
    device array, for callers that cannot allocate device memory."""
    T, k = topk_idx.shape
    d = x.shape[1]
    _contig(topk_idx, x, counts, offsets, row_offsets, perm_token, slot_to_row, X_perm)
    _check(_lib.load().moe_permute_noalloc(_p(topk_idx), _p(x), T, d, E, k, _p(counts),
                                           _p(offsets), _p(row_offsets), _p(perm_token),
                                           _p(slot_to_row), _p(X_perm), _stream(stream)),
           "moe_permute_noalloc")


def moe_expert_fwd(X, row_offsets, W_g, W_u, W_d, A, U, H, Y, ws, stream=None, row_gate=None):
    """row_gate [rows] fp32 (from moe_permute or moe_row_gates) folds each row's gate into h and y."""
    rows, d = X.shape
    E, f, _ = W_g.shape
    _contig(X, W_g, W_u, W_d, A, U, H, Y, ws, row_gate)
    _check(_lib.load().moe_expert_fwd(_p(X), _p(row_offsets), E, rows, d, f, _p(W_g), _p(W_u),
                                      _p(W_d), _p(A), _p(U), _p(H), _p(Y), _p(row_gate), _p(ws),
                                      0 if ws is None else ws.numel(), _stream(stream)),
           "moe_expert_fwd")


def moe_quantize_rows_fp8(X, rows_limit, Q, scale, stream=None):
    """Rowwise E4M3 codes (uint8) and fp32 scales of a [rows, cols] bf16 matrix."""
    X2 = X.reshape(-1, X.shape[-1])
    rows, cols = X2.shape
    _contig(X, Q, scale)
    _check(_lib.load().moe_quantize_rows_fp8(_p(X), _p(rows_limit), rows, cols, _p(Q), _p(scale),
                                             _stream(stream)), "moe_quantize_rows_fp8")


def moe_permute_fp8(xq, sx, slot_to_row, perm_token, row_offsets, Xq, sX, stream=None):
    """Codes and scales of the expert-major rows copied from those of the tokens."""
    T, d = xq.shape
    k = slot_to_row.shape[1]
    E = row_offsets.numel() - 1
    _contig(xq, sx, slot_to_row, perm_token, row_offsets, Xq, sX)
    _check(_lib.load().moe_permute_fp8(_p(xq), _p(sx), _p(slot_to_row), _p(perm_token),
                                       _p(row_offsets), T, d, E, k, _p(Xq), _p(sX),
                                       _stream(stream)), "moe_permute_fp8")


def moe_expert_fwd_fp8(Xq, sX, row_offsets, Wgq, sWg, Wuq, sWu, Wdq, sWd, A, U, H, Hq, sH, Y,
                       ws, stream=None, row_gate=None):
    rows, d = Xq.shape
    E, f, _ = Wgq.shape
    _contig(Xq, sX, Wgq, sWg, Wuq, sWu, Wdq, sWd, A, U, H, Hq, sH, Y, row_gate)
    _check(_lib.load().moe_expert_fwd_fp8(_p(Xq), _p(sX), _p(row_offsets), E, rows, d, f,
                                          _p(Wgq), _p(sWg), _p(Wuq), _p(sWu), _p(Wdq), _p(sWd),
                                          _p(A), _p(U), _p(H), _p(Hq), _p(sH), _p(Y),
                                          _p(row_gate), _p(ws), 0 if ws is None else ws.numel(),
                                          _stream(stream)),
           "moe_expert_fwd_fp8")


def moe_quantize_rows2_fp8(X0, X1, rows_limit, Q, scale, stream=None):
    """E4M3 codes of the rows [X0 | X1] under one scale per row: Q is [rows, 2 cols]."""
    rows, cols = X0.shape
    _contig(X0, X1, Q, scale)
    _check(_lib.load().moe_quantize_rows2_fp8(_p(X0), _p(X1), _p(rows_limit), rows, cols, _p(Q),
                                              _p(scale), _stream(stream)),
           "moe_quantize_rows2_fp8")


def moe_quantize_cols_fp8(X0, X1, Qt, scale, stream=None):
    """Columnwise E4M3 codes of E matrices [K0, N] (X0, or the stack of X0 over X1), written
    transposed: Qt [E, N, K] with K = K0 or 2 K0; scale [E N]."""
    X0v = X0.reshape(-1, X0.shape[-2], X0.shape[-1])
    E, K0, N = X0v.shape
    _contig(X0, X1, Qt, scale)
    _check(_lib.load().moe_quantize_cols_fp8(_p(X0), _p(X1), E, K0, N, _p(Qt), _p(scale),
                                             _stream(stream)), "moe_quantize_cols_fp8")


def moe_combine(Y_perm, topk_gate, slot_to_row, Y_shared, out, stream=None):
    """topk_gate None: the rows of Y_perm already carry their gates."""
    T, k = slot_to_row.shape
    d = Y_perm.shape[1]
    _contig(Y_perm, topk_gate, slot_to_row, Y_shared, out)
    _check(_lib.load().moe_combine(_p(Y_perm), _p(topk_gate), _p(slot_to_row), _p(Y_shared), T, d,
                                   k, _p(out), _stream(stream)), "moe_combine")


def moe_bias_update(counts, T, k, gamma, b, stream=None):
    E = counts.shape[0]
    _contig(counts, b)
    _check(_lib.load().moe_bias_update(_p(counts), E, T, k, float(gamma), _p(b), _stream(stream)),
           "moe_bias_update")


def moe_bias_update_proportional(counts, T, k, gamma, b, stream=None):
    E = counts.shape[0]
    _contig(counts, b)
    _check(_lib.load().moe_bias_update_proportional(_p(counts), E, T, k, float(gamma), _p(b),
                                                    _stream(stream)),
           "moe_bias_update_proportional")


def moe_combine_bwd(dY, Y_perm, topk_gate, slot_to_row, row_offsets, perm_token, dY_perm, dg,
                    stream=None):
    """topk_gate None: plain row copies; Y_perm and dg None: no gate gradient."""
    T, k = slot_to_row.shape
    d = dY.shape[1]
    E = row_offsets.shape[0] - 1
    _contig(dY, Y_perm, topk_gate, slot_to_row, row_offsets, perm_token, dY_perm, dg)
    _check(_lib.load().moe_combine_bwd(_p(dY), _p(Y_perm), _p(topk_gate), _p(slot_to_row),
                                       _p(row_offsets), _p(perm_token), T, d, E, k, _p(dY_perm),
                                       _p(dg), _stream(stream)), "moe_combine_bwd")


BWD_DH, BWD_DX, BWD_W, BWD_ALL = 1, 2, 4, 7  # moe_expert_bwd's parts


def moe_expert_bwd(dY, X, A, U, H, row_offsets, W_g, W_u, W_d, dX, dA, dU, dW_g, dW_u, dW_d, ws,
                   stream=None, row_gate=None, gate_part=None, parts=BWD_ALL, dl_rows=None,
                   W_r=None):
    """row_gate with gate_part [rows, f/64] fp32: the gate-folded backward; parts: which
    products run; dl_rows [rows] with W_r [E, d] fp32: the router term in dX's rows (see the
    header)."""
    rows, d = X.shape
    E, f, _ = W_g.shape
    _contig(dY, X, A, U, H, W_g, W_u, W_d, dX, dA, dU, dW_g, dW_u, dW_d, ws, row_gate, gate_part,
            dl_rows, W_r)
    _check(_lib.load().moe_expert_bwd(_p(dY), _p(X), _p(A), _p(U), _p(H), _p(row_offsets), E, rows,
                                      d, f, _p(W_g), _p(W_u), _p(W_d), _p(dX), _p(dA), _p(dU),
                                      _p(dW_g), _p(dW_u), _p(dW_d), _p(row_gate), _p(gate_part),
                                      int(parts), _p(dl_rows), _p(W_r), _p(ws),
                                      0 if ws is None else ws.numel(), _stream(stream)),
           "moe_expert_bwd")


def moe_expert_bwd_fp8(dYq, sdY, dY, X, A, U, H, row_offsets, Wdq, sWd, Wguq, sWgu, dX, dA, dU,
                       AUq, sAU, dW_g, dW_u, dW_d, ws, stream=None, dl_rows=None, W_r=None):
    """Wdq [E, f, d] and Wguq [E, d, 2f]: moe_quantize_cols_fp8 of W_d and of W_g over W_u;
    dl_rows with W_r: the router term in dX's rows (see the header)."""
    rows, d = X.shape
    E, f, _ = Wdq.shape
    _contig(dYq, sdY, dY, X, A, U, H, Wdq, sWd, Wguq, sWgu, dX, dA, dU, AUq, sAU, dW_g, dW_u,
            dW_d, ws, dl_rows, W_r)
    _check(_lib.load().moe_expert_bwd_fp8(_p(dYq), _p(sdY), _p(dY), _p(X), _p(A), _p(U), _p(H),
                                          _p(row_offsets), E, rows, d, f, _p(Wdq), _p(sWd),
                                          _p(Wguq), _p(sWgu), _p(dX), _p(dA), _p(dU), _p(AUq),
                                          _p(sAU), _p(dW_g), _p(dW_u), _p(dW_d), _p(dl_rows),
                                          _p(W_r), _p(ws), 0 if ws is None else ws.numel(),
                                          _stream(stream)),
           "moe_expert_bwd_fp8")


def moe_combine_bwd_fp8(dY, Y_perm, topk_gate, slot_to_row, row_offsets, perm_token, dY_perm,
                        dg, dYq, sdY, stream=None):
    """moe_combine_bwd plus the E4M3 codes and scales of the dY_perm rows."""
    T, k = slot_to_row.shape
    d = dY.shape[1]
    E = row_offsets.shape[0] - 1
    _contig(dY, Y_perm, topk_gate, slot_to_row, row_offsets, perm_token, dY_perm, dg, dYq, sdY)
    _check(_lib.load().moe_combine_bwd_fp8(_p(dY), _p(Y_perm), _p(topk_gate), _p(slot_to_row),
                                           _p(row_offsets), _p(perm_token), T, d, E, k,
                                           _p(dY_perm), _p(dg), _p(dYq), _p(sdY),
                                           _stream(stream)), "moe_combine_bwd_fp8")


def moe_row_gates(topk_gate, slot_to_row, row_gate, stream=None):
    T, k = topk_gate.shape
    _contig(topk_gate, slot_to_row, row_gate)
    _check(_lib.load().moe_row_gates(_p(topk_gate), _p(slot_to_row), T, k, row_gate.numel(),
                                     _p(row_gate), _stream(stream)), "moe_row_gates")


def moe_gate_grad(gate_part, slot_to_row, f, dg, stream=None):
    T, k = slot_to_row.shape
    _contig(gate_part, slot_to_row, dg)
    _check(_lib.load().moe_gate_grad(_p(gate_part), _p(slot_to_row), T, k, f, _p(dg),
                                     _stream(stream)), "moe_gate_grad")


def moe_route_bwd(dg, x, topk_idx, topk_gate, topk_score, logits, lse, E, mode, z_coef, dlogits,
                  dW_r, ws, stream=None, dlogits_extra=None, slot_to_row=None, dl_rows=None):
    """slot_to_row with dl_rows [rows] fp32: each slot's logit gradient at its row as well."""
    T, k = topk_idx.shape
    d = x.shape[1]
    _contig(dg, x, topk_idx, topk_gate, topk_score, logits, lse, dlogits, dW_r, ws, dlogits_extra,
            slot_to_row, dl_rows)
    _check(_lib.load().moe_route_bwd(_p(dg), _p(x), _p(topk_idx), _p(topk_gate), _p(topk_score),
                                     _p(logits), _p(lse), _p(dlogits_extra), T, d, E, k, mode,
                                     float(z_coef), _p(dlogits), _p(dW_r), _p(slot_to_row),
                                     _p(dl_rows), _p(ws), ws.numel(), _stream(stream)),
           "moe_route_bwd")


def moe_aux_loss(logits, topk_idx, mode, seq_len, switch_coef, seq_coef, aux_loss, aux_f, ws,
                 stream=None):
    T, E = logits.shape
    k = topk_idx.shape[1]
    _contig(logits, topk_idx, aux_loss, aux_f, ws)
    _check(_lib.load().moe_aux_loss(_p(logits), _p(topk_idx), T, E, k, mode, seq_len,
                                    float(switch_coef), float(seq_coef), _p(aux_loss), _p(aux_f),
                                    _p(ws), ws.numel(), _stream(stream)), "moe_aux_loss")


def moe_aux_loss_bwd(logits, aux_f, mode, seq_len, switch_coef, seq_coef, dlogits_aux,
                     stream=None):
    T, E = logits.shape
    _contig(logits, aux_f, dlogits_aux)
    _check(_lib.load().moe_aux_loss_bwd(_p(logits), _p(aux_f), T, E, mode, seq_len,
                                        float(switch_coef), float(seq_coef), _p(dlogits_aux),
                                        _stream(stream)), "moe_aux_loss_bwd")


def moe_permute_bwd(dX_perm, slot_to_row, dx_shared, dlogits, W_r, dx, stream=None,
                    dx_router=None):
    """dx_router [T, d] fp32 (from moe_router_dx) in place of (dlogits, W_r)."""
    T, k = slot_to_row.shape
    d = dx.shape[1]
    E = 0 if W_r is None else W_r.shape[0]
    _contig(dX_perm, slot_to_row, dx_shared, dlogits, W_r, dx, dx_router)
    _check(_lib.load().moe_permute_bwd(_p(dX_perm), _p(slot_to_row), _p(dx_shared), _p(dlogits),
                                       _p(W_r), _p(dx_router), T, d, max(E, 1), k, _p(dx),
                                       _stream(stream)),
           "moe_permute_bwd")


def moe_router_dx(dlogits, W_r, dx_r, ws, stream=None):
    """The router's input-gradient term dlogits W_r on the tensor cores (fp32 [T, d])."""
    T, E = dlogits.shape
    d = W_r.shape[1]
    _contig(dlogits, W_r, dx_r, ws)
    _check(_lib.load().moe_router_dx(_p(dlogits), _p(W_r), T, d, E, _p(dx_r), _p(ws), ws.numel(),
                                     _stream(stream)), "moe_router_dx")
