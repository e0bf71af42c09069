"""Seeded synthetic inputs for MLA decode, shared by the tests, the bench and the oracle checks.

This module draws random numbers and lays them out; it holds none of the attention
arithmetic.  Every tensor is drawn per sequence from its own ``torch.Generator``
(seeded from a stable hash of ``(seed, stream name, index)``), so any single
sequence of a large workload can be regenerated on its own for sampled checks.

Recipe (all N(0,1) draws in fp32, then rounded to bf16 with round-to-nearest-even):
  * cache rows   [T_alloc_b, 576]  per sequence b  (512 latent c^KV + 64 k^R)
  * q_nope       [S, H, 128], q_rope [S, H, 64]     per sequence b
  * W_UK, W_UV   [H, 512, 128], N(0,1) * (1/sqrt(512))
  * ragged lengths: uniform integers in [lo, hi]; pages: a seeded permutation of
    the pool's page ids, assigned in sequence order.
"""
from __future__ import annotations

import math
import zlib
from dataclasses import dataclass, field

import torch

D_C = 512
D_R = 64
D_NOPE = 128
D_V = 128
ROW = D_C + D_R
D_CQ = 1536      # query latent width of DeepSeek-V3 (the pages' module: d_c' = 1536)
D_MODEL = 4096   # model width of the pages' module


def _gen(seed: int, stream: str, index: int = 0) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(zlib.crc32(f"{seed}:{stream}:{index}".encode()) & 0x7FFFFFFF)
    return g


def randn_bf16(shape, seed: int, stream: str, index: int = 0, std: float = 1.0) -> torch.Tensor:
    x = torch.randn(*shape, generator=_gen(seed, stream, index), dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


@dataclass
class DecodeCase:
    """Shape and structure of one decode workload (no data)."""
    name: str
    B: int
    S: int
    H: int
    seqlens: list
    paged: bool = False
    page_size: int = 64
    causal: bool = False
    rope: bool = False
    theta: float = 10000.0
    num_splits: int = 0          # 0: let the library choose
    seed: int = 0
    t_cap: int = 0               # contiguous layout: rows reserved per sequence
    pages_per_seq: list = field(default_factory=list)
    block_table: torch.Tensor | None = None   # int32 [B, max_pages] (paged only)
    num_pages: int = 0

    @property
    def max_pages(self) -> int:
        return 0 if self.block_table is None else int(self.block_table.shape[1])

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(D_NOPE + D_R)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.seqlens))

    def rows_alloc(self, b: int) -> int:
        if self.paged:
            return self.pages_per_seq[b] * self.page_size
        return self.t_cap

    def q_positions(self) -> torch.Tensor:
        """Position of query token s of sequence b: the last S rows of the sequence."""
        pos = torch.empty(self.B, self.S, dtype=torch.int32)
        for b, T in enumerate(self.seqlens):
            for s in range(self.S):
                pos[b, s] = T - self.S + s
        return pos


def make_case(name: str, B: int, S: int, H: int, seqlens, *, paged=False, page_size=64,
              causal=False, rope=False, theta=10000.0, num_splits=0, seed=0, t_cap=None) -> DecodeCase:
    seqlens = [int(t) for t in seqlens]
    case = DecodeCase(name=name, B=B, S=S, H=H, seqlens=seqlens, paged=paged, page_size=page_size,
                      causal=causal, rope=rope, theta=theta, num_splits=num_splits, seed=seed)
    if paged:
        case.pages_per_seq = [max(1, -(-t // page_size)) for t in seqlens]
        case.num_pages = sum(case.pages_per_seq)
        perm = torch.randperm(case.num_pages, generator=_gen(seed, "perm"))
        max_pages = max(case.pages_per_seq)
        bt = torch.zeros(B, max_pages, dtype=torch.int32)
        off = 0
        for b, n in enumerate(case.pages_per_seq):
            bt[b, :n] = perm[off:off + n].to(torch.int32)
            off += n
        case.block_table = bt
    else:
        case.t_cap = int(t_cap if t_cap is not None else max(max(seqlens), 1))
    return case


def ragged_lengths(B: int, lo: int, hi: int, seed: int) -> list:
    return torch.randint(lo, hi + 1, (B,), generator=_gen(seed, "len")).tolist()


# The five workloads the path is built and measured on.
def tiny(seed=0):
    return make_case("tiny", 4, 1, 16, [256] * 4, seed=seed)


def dsv3(seed=0):
    return make_case("dsv3_decode", 64, 1, 128, [4096] * 64, seed=seed)


def ragged_paged(seed=0):
    return make_case("ragged_paged", 32, 1, 128, ragged_lengths(32, 512, 32768, seed),
                     paged=True, page_size=64, seed=seed)


def long_splitkv(seed=0, num_splits=0):
    return make_case("long_splitkv", 2, 1, 128, [131072] * 2, num_splits=num_splits, seed=seed)


def mtp(seed=0):
    return make_case("mtp_causal", 128, 2, 128, [8192] * 128, causal=True, rope=True, seed=seed)


WORKLOADS = {"tiny": tiny, "dsv3_decode": dsv3, "ragged_paged": ragged_paged,
             "long_splitkv": long_splitkv, "mtp_causal": mtp}


# ----------------------------------------------------------------------------
# Data
# ----------------------------------------------------------------------------

def seq_rows(case: DecodeCase, b: int) -> torch.Tensor:
    """bf16 [rows_alloc(b), 576] cache rows of sequence b (rows >= seqlens[b] are padding)."""
    return randn_bf16((case.rows_alloc(b), ROW), case.seed, "kv", b)


def seq_queries(case: DecodeCase, b: int):
    """(q_nope [S,H,128], q_rope [S,H,64]) bf16 of sequence b (q_rope unrotated)."""
    return (randn_bf16((case.S, case.H, D_NOPE), case.seed, "qn", b),
            randn_bf16((case.S, case.H, D_R), case.seed, "qr", b))


def weights(case: DecodeCase):
    """(W_UK, W_UV) bf16 [H, 512, 128], std 1/sqrt(512)."""
    std = 1.0 / math.sqrt(D_C)
    return (randn_bf16((case.H, D_C, D_NOPE), case.seed, "wuk", 0, std),
            randn_bf16((case.H, D_C, D_V), case.seed, "wuv", 0, std))


def seq_q_cat(case: DecodeCase, b: int) -> torch.Tensor:
    """bf16 [S, H, 576] query rows of sequence b in the layout the latent decode reads
    ([q~ (512) | q^R (64)]), drawn directly rather than produced by the key absorption:
    q~ ~ N(0, 1/4), the spread of q_nope W_UK^T for the draws above (128 products of
    variance 1/512 each), and q^R ~ N(0, 1)."""
    lat = randn_bf16((case.S, case.H, D_C), case.seed, "qlat", b, std=0.5)
    rope = randn_bf16((case.S, case.H, D_R), case.seed, "qcr", b)
    return torch.cat([lat, rope], dim=-1)


def q_cat(case: DecodeCase) -> torch.Tensor:
    """bf16 [B, S, H, 576]: seq_q_cat of every sequence."""
    out = torch.empty(case.B, case.S, case.H, ROW, dtype=torch.bfloat16)
    for b in range(case.B):
        out[b] = seq_q_cat(case, b)
    return out


def pool_positions(case: DecodeCase) -> torch.Tensor:
    """int32 [num_pages * page_size]: the position in its sequence of every row of a page
    pool (row r of page block_table[b, i] is position i * page_size + r of sequence b)."""
    pos = torch.zeros(case.num_pages * case.page_size, dtype=torch.int32)
    r = torch.arange(case.page_size, dtype=torch.int32)
    for b in range(case.B):
        for i in range(case.pages_per_seq[b]):
            page = int(case.block_table[b, i])
            pos[page * case.page_size:(page + 1) * case.page_size] = i * case.page_size + r
    return pos


def query_side_weights(case: DecodeCase, d_cq: int = D_CQ):
    """W_UQ bf16 [H, d_cq, 128], std 1/sqrt(d_cq) (q_nope[h] = c^Q W_UQ[h])."""
    return randn_bf16((case.H, d_cq, D_NOPE), case.seed, "wuq", 0, 1.0 / math.sqrt(d_cq))


def output_weights(case: DecodeCase, d_model: int = D_MODEL):
    """W_O bf16 [H, 128, d_model], std 1/sqrt(H*128): head h's rows of the output projection."""
    return randn_bf16((case.H, D_V, d_model), case.seed, "wo", 0, 1.0 / math.sqrt(case.H * D_V))


def seq_c_q(case: DecodeCase, b: int, d_cq: int = D_CQ) -> torch.Tensor:
    """bf16 [S, d_cq] query latents c^Q of sequence b, N(0, 1)."""
    return randn_bf16((case.S, d_cq), case.seed, "cq", b)


def c_q(case: DecodeCase, d_cq: int = D_CQ) -> torch.Tensor:
    """bf16 [B, S, d_cq]: seq_c_q of every sequence."""
    return torch.stack([seq_c_q(case, b, d_cq) for b in range(case.B)])


def queries(case: DecodeCase):
    qn = torch.empty(case.B, case.S, case.H, D_NOPE, dtype=torch.bfloat16)
    qr = torch.empty(case.B, case.S, case.H, D_R, dtype=torch.bfloat16)
    for b in range(case.B):
        qn[b], qr[b] = seq_queries(case, b)
    return qn, qr


FP8_ROW = 640   # bytes of a row of the FP8 cache: 512 E4M3 codes, then k^R as 64 bf16


def seq_fp8_rows(case: DecodeCase, b: int):
    """Sequence b's rows in the FP8 form, drawn directly (no quantizer): E4M3 codes
    uniform over the magnitude fields 0x00..0x77 (values 0 .. 240) with a random sign,
    k^R N(0,1) in bf16, one power-of-two scale per row from {2^-9, 2^-8, 2^-7}.
    Returns (uint8 [rows_alloc(b), 640], fp32 [rows_alloc(b)])."""
    n = case.rows_alloc(b)
    g = _gen(case.seed, "fp8", b)
    mag = torch.randint(0, 0x78, (n, D_C), generator=g, dtype=torch.int32)
    sign = torch.randint(0, 2, (n, D_C), generator=g, dtype=torch.int32) * 0x80
    row = torch.empty(n, FP8_ROW, dtype=torch.uint8)
    row[:, :D_C] = (mag + sign).to(torch.uint8)
    row[:, D_C:] = randn_bf16((n, D_R), case.seed, "fp8kr", b).view(torch.uint8).view(n, 2 * D_R)
    scales = torch.pow(2.0, torch.randint(-9, -6, (n,), generator=g).to(torch.float32))
    return row, scales


def fp8_cache(case: DecodeCase, device="cpu"):
    """The whole FP8 cache: (uint8 [B, t_cap, 640] or pool [num_pages, page, 640],
    fp32 scales [B, t_cap] or [num_pages, page])."""
    if case.paged:
        out = torch.zeros(case.num_pages, case.page_size, FP8_ROW, dtype=torch.uint8, device=device)
        sc = torch.ones(case.num_pages, case.page_size, dtype=torch.float32, device=device)
        for b in range(case.B):
            rows, s = seq_fp8_rows(case, b)
            ids = case.block_table[b, :case.pages_per_seq[b]].long().to(device)
            out[ids] = rows.view(-1, case.page_size, FP8_ROW).to(device)
            sc[ids] = s.view(-1, case.page_size).to(device)
        return out, sc
    out = torch.empty(case.B, case.t_cap, FP8_ROW, dtype=torch.uint8, device=device)
    sc = torch.empty(case.B, case.t_cap, dtype=torch.float32, device=device)
    for b in range(case.B):
        rows, s = seq_fp8_rows(case, b)
        out[b].copy_(rows)
        sc[b].copy_(s)
    return out, sc


def cache(case: DecodeCase, device="cpu", pin=False) -> torch.Tensor:
    """The whole cache: contiguous [B, t_cap, 576] or a page pool [num_pages, page, 576].

    Filled one sequence at a time so that only one sequence's fp32 draw is alive.
    """
    if case.paged:
        out = torch.empty(case.num_pages, case.page_size, ROW, dtype=torch.bfloat16,
                          device=device, pin_memory=pin and device == "cpu")
        for b in range(case.B):
            rows = seq_rows(case, b).view(-1, case.page_size, ROW)
            ids = case.block_table[b, :case.pages_per_seq[b]].long()
            if device == "cpu":
                out[ids] = rows
            else:
                out[ids.to(device)] = rows.to(device)
        return out
    out = torch.empty(case.B, case.t_cap, ROW, dtype=torch.bfloat16, device=device,
                      pin_memory=pin and device == "cpu")
    for b in range(case.B):
        out[b].copy_(seq_rows(case, b))
    return out
