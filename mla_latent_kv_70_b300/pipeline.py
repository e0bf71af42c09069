"""One decode step of the hot path, with its buffers allocated once.

[append the step's new latent rows to the cache, k^R rotated]  ->  absorb (q~ = q_nope
W_UK^T, RoPE'd q_rope appended)  ->  latent attention over the cache (split along the
cache and merged by log-sum-exp when planned)  ->  W_UV up-projection.  Each stage is one
call of the C ABI; nothing is computed here.
"""
from __future__ import annotations

import math

import torch

from . import (D_C, D_V, ROW, mla_absorb_q, mla_append_latent, mla_append_latent_fp8, mla_decode_latent,
               mla_decode_latent_fp8, mla_decode_num_splits, mla_decode_plan_splits,
               mla_decode_workspace_bytes, mla_out_proj_uv)


class DecodeStep:
    def __init__(self, B, S, H, w_uk, w_uv, *, max_seqlen, num_splits=0, causal=False,
                 rope_theta=10000.0, scale=None, total_rows=0, seqlens=None, rope=False, device="cuda"):
        """num_splits = 0 plans the split count: from the host-side `seqlens` when given
        (mla_decode_plan_splits), else from max_seqlen and total_rows."""
        self.B, self.S, self.H = B, S, H
        self.w_uk, self.w_uv = w_uk, w_uv
        self.max_seqlen = int(max_seqlen)
        self.causal = causal
        self.rope_theta = rope_theta
        self.rope = rope             # rotate appended k^R rows (append only)
        self.scale = scale if scale is not None else 1.0 / math.sqrt(128 + 64)
        if num_splits:
            self.num_splits = num_splits
        elif seqlens is not None:
            self.num_splits = mla_decode_plan_splits(seqlens, S, H, causal=causal, max_seqlen=self.max_seqlen)
        else:
            self.num_splits = mla_decode_num_splits(B, S, H, self.max_seqlen, total_rows)
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

    def append(self, new_rows, kv, seqlens, *, block_table=None, kv_scale=None, stream=None):
        """Add the step's latent rows [B,S,576] (k^R not yet rotated) at positions
        seqlens[b] + s and advance seqlens; rotated with this step's RoPE base when it
        applies RoPE (rope_theta > 0).  A uint8 kv is the FP8 cache: the rows are
        quantized as they are written."""
        theta = self.rope_theta if self.rope else 0.0
        if kv.dtype == torch.uint8:
            mla_append_latent_fp8(new_rows, seqlens, kv, kv_scale, rope_theta=theta, block_table=block_table,
                                  status=self.status, stream=stream)
        else:
            mla_append_latent(new_rows, seqlens, kv, rope_theta=theta, block_table=block_table,
                              status=self.status, stream=stream)

    def capture(self, q_nope, q_rope, kv, seqlens, *, block_table=None, q_pos=None, new_rows=None,
                kv_scale=None):
        """Record one step on these buffers as a CUDA graph and return a callable that
        replays it on the current stream.  The library makes no host synchronisation, so
        the step is capturable; a replay reads whatever the given tensors hold then, and
        writes self.q_cat / o_lat / lse / o.  One eager step runs first (outside the
        capture) so that one-time per-device set-up is done before capturing; with
        new_rows it appends, so seqlens has advanced by S once capture() returns."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        kw = dict(block_table=block_table, q_pos=q_pos, new_rows=new_rows, kv_scale=kv_scale)
        with torch.cuda.stream(side):
            self(q_nope, q_rope, kv, seqlens, **kw)
        torch.cuda.current_stream().wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            self(q_nope, q_rope, kv, seqlens, **kw)
        self._graph = graph          # keeps the graph (and its buffers) alive
        return graph.replay

    def __call__(self, q_nope, q_rope, kv, seqlens, *, block_table=None, q_pos=None,
                 new_rows=None, kv_scale=None, stream=None):
        """One step; with new_rows [B,S,576] the step's latent rows are appended first
        (seqlens advance by S, so max_seqlen must cover the grown sequences).  A uint8 kv
        is the FP8 form of the cache (640-byte rows) with its row scales in kv_scale."""
        if new_rows is not None:
            self.append(new_rows, kv, seqlens, block_table=block_table, kv_scale=kv_scale, stream=stream)
        mla_absorb_q(q_nope, q_rope, self.w_uk, q_pos, self.rope_theta, self.q_cat, stream)
        kw = dict(scale=self.scale, max_seqlen=self.max_seqlen, block_table=block_table, causal=self.causal,
                  num_splits=self.num_splits, workspace=self.workspace, status=self.status, stream=stream)
        if kv.dtype == torch.uint8:
            mla_decode_latent_fp8(self.q_cat, kv, kv_scale, seqlens, self.o_lat, self.lse, **kw)
        else:
            mla_decode_latent(self.q_cat, kv, seqlens, self.o_lat, self.lse, **kw)
        mla_out_proj_uv(self.o_lat, self.w_uv, self.o, stream)
        return self.o
