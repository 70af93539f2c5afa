"""The MoE layer step on one GPU, as a sequence of C-ABI calls on one stream.

Forward (route -> permute -> routed experts -> shared expert -> combine) and backward
(combine backward -> routed experts backward -> shared expert backward -> router backward
-> input gradient), then the aux-loss-free bias update. Every step runs in the library's
CUDA kernels; this module only owns the device buffers (allocated once per shape) and the
call order.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import ops


@dataclass
class MoEShape:
    T: int
    d: int
    E: int
    k: int
    f: int
    f_shared: int = 0
    mode: int = ops.MODE_SIGMOID
    z_coef: float = 0.0
    aux_switch: float = 0.0
    aux_seq: float = 0.0
    seq_len: int = 0
    fp8: bool = False        # expert forward GEMMs on E4M3 operands
    fp8_dgrad: bool = False  # and the expert backward's data-gradient GEMMs too

    @property
    def has_aux(self) -> bool:
        return self.aux_switch != 0.0 or self.aux_seq != 0.0

    @classmethod
    def from_config(cls, cfg) -> "MoEShape":
        return cls(cfg.T, cfg.d, cfg.E, cfg.k, cfg.f, cfg.f_shared, cfg.mode_id, cfg.z_coef,
                   cfg.aux_switch, cfg.aux_seq, cfg.seq_len or cfg.T,
                   cfg.precision in ("fp8", "fp8_dgrad"), cfg.precision == "fp8_dgrad")


def _empty(shape, dtype, dev):
    return torch.empty(shape, dtype=dtype, device=dev)


class MoEPlan:
    """Device buffers of one layer shape and the forward / backward call sequences."""

    # Shared-expert GEMM work per step (FLOPs, forward + backward) below which the shared
    # expert runs on a side stream. Measured on GB300: the small fine-grained layer (T 8192,
    # d 1024, shared 512: 0.08 TFLOP) 0.835 -> 0.746 ms per step with the overlap; the large
    # layer (T 65536, d 4096, shared 3072: 14.8 TFLOP) 51.3 -> 52.7 ms, as it runs at the
    # power cap, where concurrent kernels add interference and no energy budget.
    OVERLAP_SHARED_MAX_FLOPS = 1e12
    ROUTER_ROWS_MIN_FF = 768

    def __init__(self, shape: MoEShape, device="cuda", backward: bool = True,
                 overlap_shared: bool | None = None):
        s = self.s = shape
        dev = torch.device(device)
        bf, f32, i32, i64 = torch.bfloat16, torch.float32, torch.int32, torch.int64
        T, d, E, k, f, fs = s.T, s.d, s.E, s.k, s.f, s.f_shared
        R = ops.moe_padded_rows(T, k, E)
        self.R = R
        self.ws = _empty((ops.moe_workspace_bytes(T, d, E, k),), torch.uint8, dev)
        # The shared expert depends only on x (forward) and dY (backward): for small layers it
        # runs on a side stream, so that its GEMMs overlap the routed path's short kernels
        # (routing, permutation, the gradient gather, the router backward). Own scratch there.
        if overlap_shared is None:
            overlap_shared = 18.0 * T * d * fs < self.OVERLAP_SHARED_MAX_FLOPS
        self.overlap = bool(fs) and overlap_shared
        self.side = torch.cuda.Stream(dev) if self.overlap else None
        self.ws_side = (_empty((ops.moe_workspace_bytes(T, d, 1, 1),), torch.uint8, dev)
                        if self.overlap else self.ws)
        self.logits = _empty((T, E), f32, dev)
        self.topk_idx = _empty((T, k), i32, dev)
        self.topk_gate = _empty((T, k), f32, dev)
        self.topk_score = _empty((T, k), f32, dev)
        self.lse = _empty((T,), f32, dev)
        self.z_loss = torch.zeros((1,), dtype=f32, device=dev)
        self.counts = _empty((E,), i32, dev)
        self.offsets = _empty((E + 1,), i64, dev)
        self.row_offsets = _empty((E + 1,), i64, dev)
        self.perm_token = _empty((R,), i32, dev)
        self.slot_to_row = _empty((T, k), i32, dev)
        self.X_perm = _empty((R, d), bf, dev)
        self.A = _empty((R, f), bf, dev)
        self.U = _empty((R, f), bf, dev)
        self.H = _empty((R, f), bf, dev)
        self.Y_perm = _empty((R, d), bf, dev)
        # bf16 experts take each row's gate inside (g * h before the linear down projection);
        # the FP8 experts quantise the ungated h, so there the combine applies the gates
        self.fold_gate = not s.fp8
        self.row_gate = _empty((R,), f32, dev) if self.fold_gate else None
        self.out = _empty((T, d), bf, dev)
        if fs:
            self.As = _empty((T, fs), bf, dev)
            self.Us = _empty((T, fs), bf, dev)
            self.Hs = _empty((T, fs), bf, dev)
            self.Ys = _empty((T, d), bf, dev)
        if s.fp8:  # E4M3 codes and fp32 scales of every forward GEMM operand
            u8 = torch.uint8
            self.X8, self.sX = _empty((R, d), u8, dev), _empty((R,), f32, dev)
            self.H8, self.sH = _empty((R, f), u8, dev), _empty((R,), f32, dev)
            self.Wg8, self.sWg = _empty((E, f, d), u8, dev), _empty((E * f,), f32, dev)
            self.Wu8, self.sWu = _empty((E, f, d), u8, dev), _empty((E * f,), f32, dev)
            self.Wd8, self.sWd = _empty((E, d, f), u8, dev), _empty((E * d,), f32, dev)
            # codes of the token rows: copied to the expert-major rows, and the shared
            # expert's operand
            self.x8, self.sx = _empty((T, d), u8, dev), _empty((T,), f32, dev)
            if fs:
                self.Hs8, self.sHs = _empty((T, fs), u8, dev), _empty((T,), f32, dev)
                self.Wsg8, self.sWsg = _empty((1, fs, d), u8, dev), _empty((fs,), f32, dev)
                self.Wsu8, self.sWsu = _empty((1, fs, d), u8, dev), _empty((fs,), f32, dev)
                self.Wsd8, self.sWsd = _empty((1, d, fs), u8, dev), _empty((d,), f32, dev)
        if s.has_aux:
            self.aux_loss = torch.zeros((2,), dtype=f32, device=dev)
            self.aux_f = _empty((E + (T // s.seq_len) * E,), f32, dev)
        self.has_backward = backward
        self.router_rows, self.dl_rows = False, None
        if backward and s.fp8_dgrad:  # E4M3 operands of the data-gradient GEMMs
            u8 = torch.uint8
            self.dYq, self.sdY = _empty((R, d), u8, dev), _empty((R,), f32, dev)
            self.AUq, self.sAU = _empty((R, 2 * f), u8, dev), _empty((R,), f32, dev)
            self.Wdq_t, self.sWd_t = _empty((E, f, d), u8, dev), _empty((E * f,), f32, dev)
            self.Wguq_t, self.sWgu_t = _empty((E, d, 2 * f), u8, dev), _empty((E * d,), f32, dev)
            if fs:
                self.dYsq, self.sdYs = _empty((T, d), u8, dev), _empty((T,), f32, dev)
                self.AUsq, self.sAUs = _empty((T, 2 * fs), u8, dev), _empty((T,), f32, dev)
                self.Wsdq_t, self.sWsd_t = _empty((1, fs, d), u8, dev), _empty((fs,), f32, dev)
                self.Wsguq_t, self.sWsgu_t = (_empty((1, d, 2 * fs), u8, dev),
                                              _empty((d,), f32, dev))
        if backward:
            if s.has_aux:
                self.dlogits_aux = _empty((T, E), f32, dev)
            self.dY_perm = _empty((R, d), bf, dev)
            self.dg = _empty((T, k), f32, dev)
            if self.fold_gate:  # gate-gradient partial sums of the expert backward
                self.gate_part = _empty((R, f // 64), f32, dev)
            self.dA = _empty((R, f), bf, dev)
            self.dU = _empty((R, f), bf, dev)
            self.dX_perm = _empty((R, d), bf, dev)
            self.dW_g = _empty((E, f, d), bf, dev)
            self.dW_u = _empty((E, f, d), bf, dev)
            self.dW_d = _empty((E, d, f), bf, dev)
            self.dlogits = _empty((T, E), f32, dev)
            # dense logit gradients (softmax router, balancing losses): the router's input-
            # gradient term runs on the tensor cores instead of in the dx kernel's row loop
            self.router_dx_tc = (s.mode == ops.MODE_SOFTMAX or s.has_aux) and E <= 128
            # sigmoid routing without balancing losses: a token's logit gradient is zero off
            # its chosen experts, so its router input-gradient term dl[t, e] W_r[e] joins
            # each chosen slot's dX row in the data-gradient GEMM's epilogue, and the token
            # sum reads no fp32 W_r rows (large layer: 1.05 -> 0.80 ms for the token sum).
            # That GEMM's reduction is K = 2 d_ff; below ROUTER_ROWS_MIN_FF its epilogue sets
            # its pace and the term costs more there than it saves (small fine-grained
            # layer, d_ff 256: 0.675 -> 0.681 ms per step), so short experts keep the term
            # in the token sum.
            self.router_rows = (s.mode == ops.MODE_SIGMOID and not s.has_aux
                                and s.f >= self.ROUTER_ROWS_MIN_FF)
            self.dl_rows = torch.zeros((R,), dtype=f32, device=dev) if self.router_rows else None
            self.dx_r = _empty((T, d), f32, dev) if self.router_dx_tc else None
            self.dW_r = _empty((E, d), f32, dev)
            self.dx = _empty((T, d), bf, dev)
            if fs:
                self.dAs = _empty((T, fs), bf, dev)
                self.dUs = _empty((T, fs), bf, dev)
                self.dxs = _empty((T, d), bf, dev)
                self.dWs_g = _empty((fs, d), bf, dev)
                self.dWs_u = _empty((fs, d), bf, dev)
                self.dWs_d = _empty((d, fs), bf, dev)

    # Optional list that receives (start, end) CUDA event pairs around every grouped-GEMM
    # entry point call, recorded on the launching stream (used to time the GEMMs inside a
    # step without adding synchronisation).
    gemm_events = None

    def _gemm(self, fn, *args, stream=None, **kw):
        if self.gemm_events is None:
            fn(*args, stream, **kw)
            return
        st = stream if stream is not None else torch.cuda.current_stream()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        fn(*args, stream, **kw)
        b.record(st)
        self.gemm_events.append((a, b))

    def launches_per_step(self, backward=True, bias_update=False) -> int:
        """Kernel launches of one step through this plan (what the entry points enqueue)."""
        s = self.s
        n = 1 + (1 if s.E <= 128 else 0)                   # route (W_r pieces + tensor-core
        n += 1 if s.mode == ops.MODE_SOFTMAX else 0         # logits) (+ z-loss reduction)
        if s.has_aux:
            n += 2 + (1 if backward else 0)                 # balancing losses (+ gradient)
        n += 4                                              # permute (the padding rows and
                                                            # folded row gates in the scatter)
        if s.fp8:  # quantise x, W_g, W_u, W_d; expert-major codes (2); G1, quantise H, G2
            n += 9 + (6 if s.f_shared else 0)               # (shared: its weights, G1, H, G2)
        else:
            n += 2 + (2 if s.f_shared else 0)               # expert forward (G1, G2)
        n += 1                                              # combine
        if backward:
            n += 1                                          # combine backward (+ padding rows)
            n += 1 if not s.fp8 else 0                      # gate gradient from its partials
            if s.fp8_dgrad:  # pad the dY codes, W_d and W_g/W_u columns (3 each), B2,
                n += 13 + (12 if s.f_shared else 0)         # [dA|dU] rows, B4, order, B3, B5
                                                            # (shared: quantise dY rows)
            else:
                n += 5 + (4 if s.f_shared else 0)           # expert backward (+ expert order)
            n += 3                                          # router backward
            if (s.mode == ops.MODE_SOFTMAX or s.has_aux) and s.E <= 128:
                n += 3                                      # router dx: two splits + GEMM
            n += 1                                          # input gradient
        if bias_update:
            n += 1
        return n

    # ------------------------------------------------------------------ forward
    def forward(self, x, W_r, b, W_g, W_u, W_d, Ws_g=None, Ws_u=None, Ws_d=None, stream=None):
        s = self.s
        self.x = x
        self.W = (W_r, b, W_g, W_u, W_d, Ws_g, Ws_u, Ws_d)
        softmax = s.mode == ops.MODE_SOFTMAX
        main = stream if stream is not None else torch.cuda.current_stream()
        if s.fp8:  # before the fork: the routed rows and the shared expert both use them
            ops.moe_quantize_rows_fp8(x, None, self.x8, self.sx, stream)
        if s.f_shared and self.overlap:  # fork: the shared expert on the side stream
            self.side.wait_stream(main)
            self._shared_forward(x, Ws_g, Ws_u, Ws_d, self.side)
        ops.moe_route(x, W_r, None if softmax else b, s.k, s.mode, s.z_coef, self.logits,
                      self.topk_idx, self.topk_gate, self.topk_score,
                      self.lse if softmax else None, self.z_loss if softmax else None, self.ws,
                      stream)
        if s.has_aux:
            ops.moe_aux_loss(self.logits, self.topk_idx, s.mode, s.seq_len, s.aux_switch,
                             s.aux_seq, self.aux_loss, self.aux_f, self.ws, stream)
        # the combine's gate weights move before the (linear) down projection: the routed
        # experts emit g * y directly, and the combine adds rows without weights; the
        # dispatch copies each slot's gate to its row as it places the row
        ops.moe_permute(self.topk_idx, x, s.E, self.counts, self.offsets, self.row_offsets,
                        self.perm_token, self.slot_to_row, self.X_perm, self.ws, stream,
                        topk_gate=self.topk_gate if self.fold_gate else None,
                        row_gate=self.row_gate)
        ys = None
        if s.fp8:
            q = ops.moe_quantize_rows_fp8
            q(W_g, None, self.Wg8, self.sWg, stream)
            q(W_u, None, self.Wu8, self.sWu, stream)
            q(W_d, None, self.Wd8, self.sWd, stream)
            ops.moe_permute_fp8(self.x8, self.sx, self.slot_to_row, self.perm_token,
                                self.row_offsets, self.X8, self.sX, stream)
            self._gemm(ops.moe_expert_fwd_fp8, self.X8, self.sX, self.row_offsets, self.Wg8,
                       self.sWg, self.Wu8, self.sWu, self.Wd8, self.sWd, self.A, self.U, self.H,
                       self.H8, self.sH, self.Y_perm, self.ws, stream=stream)
        else:
            self._gemm(ops.moe_expert_fwd, self.X_perm, self.row_offsets, W_g, W_u, W_d, self.A,
                       self.U, self.H, self.Y_perm, self.ws, stream=stream, row_gate=self.row_gate)
        if s.f_shared:
            if self.overlap:  # join
                main.wait_stream(self.side)
            else:
                self._shared_forward(x, Ws_g, Ws_u, Ws_d, stream)
            ys = self.Ys
        ops.moe_combine(self.Y_perm, None if self.fold_gate else self.topk_gate, self.slot_to_row,
                        ys, self.out, stream)
        return self.out

    def _shared_forward(self, x, Ws_g, Ws_u, Ws_d, side):
        """The shared expert's forward on stream `side` (every token, weight 1)."""
        if self.s.fp8:
            q = ops.moe_quantize_rows_fp8
            q(Ws_g, None, self.Wsg8, self.sWsg, side)
            q(Ws_u, None, self.Wsu8, self.sWsu, side)
            q(Ws_d, None, self.Wsd8, self.sWsd, side)
            self._gemm(ops.moe_expert_fwd_fp8, self.x8, self.sx, None, self.Wsg8, self.sWsg,
                       self.Wsu8, self.sWsu, self.Wsd8, self.sWsd, self.As, self.Us, self.Hs,
                       self.Hs8, self.sHs, self.Ys, self.ws_side, stream=side)
        else:
            self._gemm(ops.moe_expert_fwd, x, None, Ws_g[None], Ws_u[None], Ws_d[None],
                       self.As, self.Us, self.Hs, self.Ys, self.ws_side, stream=side)

    # ----------------------------------------------------------------- backward
    def backward(self, dY, stream=None):
        s = self.s
        x = self.x
        W_r, b, W_g, W_u, W_d, Ws_g, Ws_u, Ws_d = self.W
        main = stream if stream is not None else torch.cuda.current_stream()
        if s.f_shared and self.overlap:  # fork: the shared expert's backward on the side stream
            self.side.wait_stream(main)
            self._shared_backward(dY, x, Ws_g, Ws_u, Ws_d, self.side)
        if self.fold_gate:
            # gate folded into the experts: dY_perm holds plain copies of the token gradients,
            # the expert backward applies each row's gate and sums the gate's gradient in parts
            ops.moe_combine_bwd(dY, None, None, self.slot_to_row, self.row_offsets,
                                self.perm_token, self.dY_perm, None, stream)
            # with the router term in the rows, dX and the weight gradients wait for the
            # logit gradient (below); the gate's gradient comes from the dh pass alone
            self._gemm(ops.moe_expert_bwd, self.dY_perm, self.X_perm, self.A, self.U, self.H,
                       self.row_offsets, W_g, W_u, W_d, self.dX_perm, self.dA, self.dU,
                       self.dW_g, self.dW_u, self.dW_d, self.ws, stream=stream,
                       row_gate=self.row_gate, gate_part=self.gate_part,
                       parts=ops.BWD_DH if self.router_rows else ops.BWD_ALL)
            ops.moe_gate_grad(self.gate_part, self.slot_to_row, s.f, self.dg, stream)
        elif s.fp8_dgrad:  # the combine backward also writes the codes of the rows it stores
            ops.moe_combine_bwd_fp8(dY, self.Y_perm, self.topk_gate, self.slot_to_row,
                                    self.row_offsets, self.perm_token, self.dY_perm, self.dg,
                                    self.dYq, self.sdY, stream)
            ops.moe_quantize_cols_fp8(W_d, None, self.Wdq_t, self.sWd_t, stream)
            ops.moe_quantize_cols_fp8(W_g, W_u, self.Wguq_t, self.sWgu_t, stream)
            if self.router_rows:  # the gate gradient is known: the logit gradient first
                self._route_bwd(x, None, stream)
            self._gemm(ops.moe_expert_bwd_fp8, self.dYq, self.sdY, self.dY_perm, self.X_perm,
                       self.A, self.U, self.H, self.row_offsets, self.Wdq_t, self.sWd_t,
                       self.Wguq_t, self.sWgu_t, self.dX_perm, self.dA, self.dU, self.AUq,
                       self.sAU, self.dW_g, self.dW_u, self.dW_d, self.ws, stream=stream,
                       dl_rows=self.dl_rows, W_r=W_r if self.router_rows else None)
        else:
            ops.moe_combine_bwd(dY, self.Y_perm, self.topk_gate, self.slot_to_row,
                                self.row_offsets, self.perm_token, self.dY_perm, self.dg, stream)
            self._gemm(ops.moe_expert_bwd, self.dY_perm, self.X_perm, self.A, self.U, self.H,
                       self.row_offsets, W_g, W_u, W_d, self.dX_perm, self.dA, self.dU,
                       self.dW_g, self.dW_u, self.dW_d, self.ws, stream=stream,
                       parts=ops.BWD_DH if self.router_rows else ops.BWD_ALL)
        dxs = None
        extra = None
        if s.has_aux:
            ops.moe_aux_loss_bwd(self.logits, self.aux_f, s.mode, s.seq_len, s.aux_switch,
                                 s.aux_seq, self.dlogits_aux, stream)
            extra = self.dlogits_aux
        rows = self.router_rows
        if not (rows and s.fp8_dgrad):  # (the FP8 path formed the logit gradient above)
            self._route_bwd(x, extra, stream)
        if rows and not s.fp8_dgrad:
            self._gemm(ops.moe_expert_bwd, self.dY_perm, self.X_perm, self.A, self.U, self.H,
                       self.row_offsets, W_g, W_u, W_d, self.dX_perm, self.dA, self.dU,
                       self.dW_g, self.dW_u, self.dW_d, self.ws, stream=stream,
                       parts=ops.BWD_DX | ops.BWD_W, dl_rows=self.dl_rows, W_r=W_r)
        if s.f_shared:
            if self.overlap:  # join
                main.wait_stream(self.side)
            else:
                self._shared_backward(dY, x, Ws_g, Ws_u, Ws_d, stream)
            dxs = self.dxs
        if self.router_dx_tc:
            ops.moe_router_dx(self.dlogits, W_r, self.dx_r, self.ws, stream)
            ops.moe_permute_bwd(self.dX_perm, self.slot_to_row, dxs, None, None, self.dx, stream,
                                dx_router=self.dx_r)
        elif rows:  # the router term is already in the rows
            ops.moe_permute_bwd(self.dX_perm, self.slot_to_row, dxs, None, None, self.dx, stream)
        else:
            ops.moe_permute_bwd(self.dX_perm, self.slot_to_row, dxs, self.dlogits, W_r, self.dx,
                                stream)
        return self.dx

    def _route_bwd(self, x, extra, stream):
        s = self.s
        softmax = s.mode == ops.MODE_SOFTMAX
        rows = self.router_rows
        ops.moe_route_bwd(self.dg, x, self.topk_idx, self.topk_gate, self.topk_score,
                          self.logits if softmax else None, self.lse if softmax else None, s.E,
                          s.mode, s.z_coef, self.dlogits, self.dW_r, self.ws, stream,
                          dlogits_extra=extra, slot_to_row=self.slot_to_row if rows else None,
                          dl_rows=self.dl_rows)

    def _shared_backward(self, dY, x, Ws_g, Ws_u, Ws_d, st):
        if self.s.fp8_dgrad:
            ops.moe_quantize_rows_fp8(dY, None, self.dYsq, self.sdYs, st)
            ops.moe_quantize_cols_fp8(Ws_d[None], None, self.Wsdq_t, self.sWsd_t, st)
            ops.moe_quantize_cols_fp8(Ws_g[None], Ws_u[None], self.Wsguq_t, self.sWsgu_t, st)
            self._gemm(ops.moe_expert_bwd_fp8, self.dYsq, self.sdYs, dY, x, self.As, self.Us,
                       self.Hs, None, self.Wsdq_t, self.sWsd_t, self.Wsguq_t, self.sWsgu_t,
                       self.dxs, self.dAs, self.dUs, self.AUsq, self.sAUs, self.dWs_g[None],
                       self.dWs_u[None], self.dWs_d[None], self.ws_side, stream=st)
            return
        self._gemm(ops.moe_expert_bwd, dY, x, self.As, self.Us, self.Hs, None, Ws_g[None],
                   Ws_u[None], Ws_d[None], self.dxs, self.dAs, self.dUs, self.dWs_g[None],
                   self.dWs_u[None], self.dWs_d[None], self.ws_side, stream=st)

    def bias_update(self, b, gamma, rule="sign", stream=None):
        if rule == "proportional":
            ops.moe_bias_update_proportional(self.counts, self.s.T, self.s.k, gamma, b, stream)
        else:
            ops.moe_bias_update(self.counts, self.s.T, self.s.k, gamma, b, stream)

    def capture_step(self, x, weights: dict, dY=None, b=None, gamma=0.0, rule="sign",
                     bias_update=False, warmup=1):
        """Record one whole step (forward, backward when dY is given, bias update) into a
        CUDA graph over this plan's fixed buffers; ``graph.replay()`` then re-runs it with
        one launch from the host. Inputs are read from the same device tensors at replay
        time, so callers refresh them in place. The warm-up runs load every kernel first."""
        W = (weights["W_r"], b, weights["W_g"], weights["W_u"], weights["W_d"],
             weights.get("Ws_g"), weights.get("Ws_u"), weights.get("Ws_d"))

        def step():
            self.forward(x, *W)
            if dY is not None:
                self.backward(dY)
                if bias_update:
                    self.bias_update(b, gamma, rule)

        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(warmup):
                step()
        torch.cuda.current_stream().wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        return graph

    def grads(self) -> dict:
        g = {"dx": self.dx, "dW_r": self.dW_r, "dW_g": self.dW_g, "dW_u": self.dW_u,
             "dW_d": self.dW_d}
        if self.s.f_shared:
            g.update(dWs_g=self.dWs_g, dWs_u=self.dWs_u, dWs_d=self.dWs_d)
        return g


class _MoEFunction(torch.autograd.Function):
    """One layer step as an autograd node over a plan's fixed buffers.

    The plan keeps the forward's activations for the backward, so a later forward through
    the same plan (the same token count) overwrites them: ``plan.generation`` counts the
    forwards and the backward refuses a stale one."""

    @staticmethod
    def forward(ctx, x, W_r, b, W_g, W_u, W_d, Ws_g, Ws_u, Ws_d, plan):
        ctx.plan = plan
        plan.generation += 1
        ctx.generation = plan.generation
        out = plan.forward(x.contiguous(), W_r, b, W_g, W_u, W_d, Ws_g, Ws_u, Ws_d)
        return out.clone()

    @staticmethod
    def backward(ctx, dY):
        plan = ctx.plan
        if plan.generation != ctx.generation:
            raise RuntimeError(
                "MoELayer: another forward with the same token count ran after this one and "
                "overwrote its saved activations; run each backward before the next forward")
        plan.backward(dY.to(torch.bfloat16).contiguous())
        g = plan.grads()
        shared = plan.s.f_shared > 0
        return (g["dx"].clone(), g["dW_r"].clone(), None, g["dW_g"].clone(), g["dW_u"].clone(),
                g["dW_d"].clone(), g["dWs_g"].clone() if shared else None,
                g["dWs_u"].clone() if shared else None, g["dWs_d"].clone() if shared else None,
                None)


class MoELayer(torch.nn.Module):
    """Fine-grained MoE layer module (bf16 experts, fp32 router and bias) on one GPU.

    ``forward(x)`` takes x [T, d] bf16 and returns out [T, d] bf16; gradients flow to x and
    every weight. The router's own losses (the z-loss in softmax mode, the balancing losses
    when their coefficients are set) enter the training loss with weight 1: their gradient
    is added in the layer's backward, and their values are read with ``z_loss()`` and
    ``aux_loss()`` for logging. The bias is a buffer: it gets no gradient and moves only by
    ``update_bias()``, called after backward with that step's expert counts.

    One plan (set of device buffers) is kept per token count; each backward must run before
    the next forward with the same token count."""

    def __init__(self, d, E, k, f, f_shared=0, mode="sigmoid", z_coef=0.0, gamma=1e-3,
                 device="cuda", bias_rule="sign", aux_switch=0.0, aux_seq=0.0, seq_len=0,
                 precision="bf16"):
        super().__init__()
        if mode not in ("sigmoid", "softmax") or bias_rule not in ("sign", "proportional") \
                or precision not in ("bf16", "fp8", "fp8_dgrad"):
            raise ValueError("mode is sigmoid or softmax, bias_rule sign or proportional, "
                             "precision bf16, fp8 or fp8_dgrad")
        self.d, self.E, self.k, self.f, self.f_shared = d, E, k, f, f_shared
        self.mode = ops.MODE_SIGMOID if mode == "sigmoid" else ops.MODE_SOFTMAX
        self.z_coef, self.gamma, self.bias_rule = z_coef, gamma, bias_rule
        self.aux_switch, self.aux_seq, self.seq_len = aux_switch, aux_seq, seq_len
        self.fp8 = precision in ("fp8", "fp8_dgrad")
        self.fp8_dgrad = precision == "fp8_dgrad"
        bf = dict(dtype=torch.bfloat16, device=device)
        self.W_r = torch.nn.Parameter(torch.randn(E, d, device=device) * d ** -0.5)
        self.register_buffer("b", torch.zeros(E, device=device))
        self.W_g = torch.nn.Parameter((torch.randn(E, f, d, device=device) * d ** -0.5).to(**bf))
        self.W_u = torch.nn.Parameter((torch.randn(E, f, d, device=device) * d ** -0.5).to(**bf))
        self.W_d = torch.nn.Parameter((torch.randn(E, d, f, device=device) * f ** -0.5).to(**bf))
        if f_shared:
            self.Ws_g = torch.nn.Parameter((torch.randn(f_shared, d, device=device) * d ** -0.5).to(**bf))
            self.Ws_u = torch.nn.Parameter((torch.randn(f_shared, d, device=device) * d ** -0.5).to(**bf))
            self.Ws_d = torch.nn.Parameter((torch.randn(d, f_shared, device=device) * f_shared ** -0.5).to(**bf))
        else:
            self.Ws_g = self.Ws_u = self.Ws_d = None
        self._plans = {}
        self._last_plan = None

    def _plan(self, T):
        if T not in self._plans:
            shape = MoEShape(T, self.d, self.E, self.k, self.f, self.f_shared, self.mode,
                             self.z_coef, self.aux_switch, self.aux_seq, self.seq_len or T,
                             self.fp8, self.fp8_dgrad)
            plan = MoEPlan(shape, self.W_g.device)
            plan.generation = 0
            self._plans[T] = plan
        return self._plans[T]

    def forward(self, x):
        if x.dim() != 2 or x.shape[1] != self.d or x.dtype != torch.bfloat16:
            raise ValueError(f"x must be [T, {self.d}] bf16, got {tuple(x.shape)} {x.dtype}")
        plan = self._plan(x.shape[0])
        self._last_plan = plan
        return _MoEFunction.apply(x, self.W_r, self.b, self.W_g, self.W_u, self.W_d, self.Ws_g,
                                  self.Ws_u, self.Ws_d, plan)

    @torch.no_grad()
    def update_bias(self):
        if self.mode == ops.MODE_SIGMOID and self._last_plan is not None:
            self._last_plan.bias_update(self.b, self.gamma, self.bias_rule)

    def z_loss(self):
        """The last forward's router z-loss ([1] fp32 device tensor; softmax mode)."""
        return None if self._last_plan is None else self._last_plan.z_loss

    def aux_loss(self):
        """The last forward's balancing losses ([2] fp32: Switch-style, sequence-wise)."""
        p = self._last_plan
        return None if p is None or not p.s.has_aux else p.aux_loss
