"""One decode step of the hot path, with its buffers allocated once.

absorb (q~ = q_nope W_UK^T, RoPE'd q_rope appended)  ->  latent attention over the
cache (split along the cache and merged by log-sum-exp when planned)  ->  W_UV
up-projection.  Each stage is one call of the C ABI; nothing is computed here.
"""
from __future__ import annotations

import math

import torch

from . import (D_C, D_V, ROW, mla_absorb_q, mla_decode_latent, mla_decode_num_splits,
               mla_decode_workspace_bytes, mla_out_proj_uv)


class DecodeStep:
    def __init__(self, B, S, H, w_uk, w_uv, *, max_seqlen, num_splits=0, causal=False,
                 rope_theta=10000.0, scale=None, total_rows=0, device="cuda"):
        self.B, self.S, self.H = B, S, H
        self.w_uk, self.w_uv = w_uk, w_uv
        self.max_seqlen = int(max_seqlen)
        self.causal = causal
        self.rope_theta = rope_theta
        self.scale = scale if scale is not None else 1.0 / math.sqrt(128 + 64)
        self.num_splits = num_splits or mla_decode_num_splits(B, S, H, self.max_seqlen, total_rows)
        ws = mla_decode_workspace_bytes(B, S, H, self.num_splits, self.max_seqlen)
        self.workspace = torch.empty(ws // 4, dtype=torch.float32, device=device) if ws else None
        self.q_cat = torch.empty(B, S, H, ROW, dtype=torch.bfloat16, device=device)
        self.o_lat = torch.empty(B, S, H, D_C, dtype=torch.float32, device=device)
        self.lse = torch.empty(B, S, H, dtype=torch.float32, device=device)
        self.o = torch.empty(B, S, H, D_V, dtype=torch.float32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    @property
    def kernels_per_step(self) -> int:
        return 3 + (1 if self.num_splits > 1 else 0)

    def __call__(self, q_nope, q_rope, kv, seqlens, *, block_table=None, q_pos=None,
                 stream=None):
        mla_absorb_q(q_nope, q_rope, self.w_uk, q_pos, self.rope_theta, self.q_cat, stream)
        mla_decode_latent(self.q_cat, kv, seqlens, self.o_lat, self.lse, scale=self.scale,
                          max_seqlen=self.max_seqlen, block_table=block_table,
                          causal=self.causal, num_splits=self.num_splits,
                          workspace=self.workspace, status=self.status, stream=stream)
        mla_out_proj_uv(self.o_lat, self.w_uv, self.o, stream)
        return self.o
