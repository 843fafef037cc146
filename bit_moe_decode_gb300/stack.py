"""A stack of routed-expert layers run in sequence through the C ABI: the whole routed-expert path of a
DeepSeek-V4-Flash-shaped model for decode and verify ("Mixed-precision compression of DeepSeek-V4-Flash",
"The recipe": 43 layers x 256 experts, top-6; "quant surgery", section 4: the first layers route by a token-id
hash table, tid2eid).

Per layer L of a call with T tokens (1 <= T <= 8):
  hash layers (L < n_hash):  moe_route_topk in hash mode (idx = tid2eid[token id], w = 1/k), then
                             moe_expert_ffn_verify;
  softmax layers:            moe_route_expert_ffn (router top-k and FFN in one launch);
  with shared experts:       moe_expert_ffn_verify on the layer's one-expert Q8_0 layer (idx 0, w 1), accumulating
                             into y (the recipe of "Mixed-precision compression of DeepSeek-V4-Flash" keeps each
                             layer's always-on shared expert in 8 bits);
  then                       moe_rms_norm_bf16: layer L + 1's x = bf16(y_L / rms(y_L)).
The model normalises the hidden state before each MoE layer; without it a stack of random layers drifts (the FFN
maps an activation of rms r to about c r^2, so the chain collapses to zero, where every router sees ties, or
overflows). There is no attention or residual in between (not on the routed-expert path). Everything here only
orders library calls on one stream; all arithmetic runs in the library's kernels.
"""
from __future__ import annotations

import torch

from . import (MOE_FMT_MXFP4, MOE_FMT_Q8_0, MOE_LAYOUT_TC, Layer, moe_expert_ffn_verify, moe_rms_norm_bf16,
               moe_route_expert_ffn, moe_route_topk)

NORM_EPS = 1e-6


class RoutedStack:
    """n_layers MXFP4 layers in the tensor-core layout (H, I, E experts each), hash routing in the first n_hash.

    Buffers (device): x[L] bf16 [T_max, H] for L = 0..n_layers (x[0] is the default input, x[L + 1] the normalised
    output of layer L), idx[L] int32 / w[L] fp32 [T_max, k] (the routing each layer used), y[L] fp32 [T_max, H] (each layer's
    fp32 output), one shared workspace (the calls run one after another on the stream)."""

    def __init__(self, H: int, I: int, E: int, k: int, n_layers: int, n_hash: int, vocab: int, T_max: int = 8,
                 device="cuda", shared_I: int = 0):
        assert 0 <= n_hash <= n_layers and 1 <= T_max <= 8
        self.H, self.I, self.E, self.k, self.n, self.n_hash, self.vocab, self.T_max = \
            H, I, E, k, n_layers, n_hash, vocab, T_max
        self.layers = [Layer(MOE_FMT_MXFP4, H, I, E, layout=MOE_LAYOUT_TC, device=device) for _ in range(n_layers)]
        self.router = [None] * n_layers          # fp16 bits [E, H] (int16 tensors) of the softmax layers
        self.tid2eid = [None] * n_layers         # int32 [vocab, k] of the hash layers
        self.x = [torch.zeros((T_max, H), dtype=torch.int16, device=device) for _ in range(n_layers + 1)]
        self.idx = [torch.zeros((T_max, k), dtype=torch.int32, device=device) for _ in range(n_layers)]
        self.w = [torch.zeros((T_max, k), dtype=torch.float32, device=device) for _ in range(n_layers)]
        self.y = [torch.zeros((T_max, H), dtype=torch.float32, device=device) for _ in range(n_layers)]
        self.ws = self.layers[0].workspace(T_max, k) if n_layers else None
        # optional shared experts: one Q8_0 expert per layer (intermediate size shared_I) and their own workspace
        self.shared = [Layer(MOE_FMT_Q8_0, H, shared_I, 1, device=device) for _ in range(n_layers)] if shared_I else []
        self.ws_shared = self.shared[0].workspace(T_max, 1) if self.shared else None
        self.one_idx = torch.zeros((T_max, 1), dtype=torch.int32, device=device)
        self.one_w = torch.ones((T_max, 1), dtype=torch.float32, device=device)

    def packed_bytes(self, shared: bool = False) -> int:
        mats = self.layers + (self.shared if shared else [])
        return sum(L.gate_up.numel() + L.down.numel() for L in mats)

    def run(self, T: int, token_ids=None, x0=None, stream=None, shared: bool = None):
        """One decode (T = 1) or verify (T <= 8) pass of T tokens through every layer: the first layer reads x0
        (bf16 [T, H], device) or, if None, x[0][:T]. token_ids (int32 [T], device) is needed when the stack has
        hash layers. shared (default: whether the stack has shared experts) adds each layer's shared expert."""
        assert 1 <= T <= self.T_max
        use_shared = bool(self.shared) if shared is None else (bool(shared) and bool(self.shared))
        for L in range(self.n):
            xin = x0 if (L == 0 and x0 is not None) else self.x[L][:T]
            xout = self.x[L + 1][:T]
            idx, w = self.idx[L][:T], self.w[L][:T]
            if L < self.n_hash:
                moe_route_topk(None, None, T, self.H, self.E, self.k, token_ids, self.tid2eid[L], self.vocab, idx, w,
                               stream=stream)
                moe_expert_ffn_verify(self.layers[L], xin, T, idx, w, self.k, self.y[L][:T], None, False, self.ws,
                                      stream=stream)
            else:
                moe_route_expert_ffn(self.layers[L], self.router[L], xin, T, self.k, idx, w, self.y[L][:T], None,
                                     False, self.ws, stream=stream)
            if use_shared:
                moe_expert_ffn_verify(self.shared[L], xin, T, self.one_idx[:T], self.one_w[:T], 1, self.y[L][:T],
                                      None, True, self.ws_shared, stream=stream)
            moe_rms_norm_bf16(self.y[L][:T], T, self.H, NORM_EPS, xout, stream=stream)

    def launches_per_run(self, shared: bool = False) -> int:
        return 2 * self.n_hash + (self.n - self.n_hash) + self.n + (self.n if shared and self.shared else 0)
