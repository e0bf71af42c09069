"""MLA decode with weight absorption on B300: Python binding of libmla.so.

The functions below carry the names of the C ABI in include/mla.h and only marshal
arguments (torch CUDA tensors -> device pointers, shapes -> ints, the current CUDA
stream).  Every step of the computation runs in the library's CUDA kernels; there is
no CPU or PyTorch fallback: a missing or unloadable libmla.so raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import inputs  # noqa: F401  (seeded synthetic inputs; no attention math)

D_C, D_R, D_NOPE, D_V, ROW = 512, 64, 128, 128, 576
MAX_SPLITS = 128

STATUS = {0: "MLA_OK", 1: "MLA_ERR_INVALID", 2: "MLA_ERR_UNSUPPORTED", 3: "MLA_ERR_CUDA",
          4: "MLA_ERR_WORKSPACE", 5: "MLA_ERR_BLOCK_TABLE", 6: "MLA_ERR_TIMEOUT"}
FLAG_BLOCK_TABLE = 1 << 5
FLAG_TIMEOUT = 1 << 6

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmla.so")

# (name, restype, argtypes) of every exported symbol.
_P, _I, _I64, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "mla_status_string": (ctypes.c_char_p, [_I]),
    "mla_device_sm_count": (_I, []),
    "mla_absorb_q": (_I, [_P, _P, _P, _P, _F, _I, _I, _I, _P, _P]),
    "mla_decode_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "mla_decode_num_splits": (_I, [_I, _I, _I, _I, _I64]),
    "mla_decode_plan_splits": (_I, [_P, _I, _I, _I, _I, _I]),
    "mla_decode_latent": (_I, [_P, _P, _I64, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I,
                               _P, _P, _P, _SZ, _P, _P]),
    "mla_decode_latent_fp8": (_I, [_P, _P, _P, _I64, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I,
                                   _P, _P, _P, _SZ, _P, _P]),
    "mla_quantize_fp8": (_I, [_P, _I64, _I64, _P, _P, _P]),
    "mla_append_latent_fp8": (_I, [_P, _I, _I, _F, _P, _P, _P, _I64, _P, _I, _I, _I, _P, _P]),
    "mla_decode_latent_noalloc": (_I, [_P, _P, _I64, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I,
                                       _I, _P, _P, _P, _P]),
    "mla_combine_partials": (_I, [_P, _P, _I, _I64, _P, _P, _P]),
    "mla_out_proj_uv": (_I, [_P, _P, _I, _I, _I, _P, _P]),
    "mla_rope_inplace": (_I, [_P, _I64, _I64, _I, _P, _F, _P]),
    "mla_debug_inject_timeout": (_I, [_I, ctypes.c_double]),
    "mla_append_latent": (_I, [_P, _I, _I, _F, _P, _P, _I64, _P, _I, _I, _I, _P, _P]),
    "mla_fuse_weights": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _P]),
    "mla_absorb_q_fused": (_I, [_P, _P, _P, _P, _F, _I, _I, _I, _I, _P, _P]),
    "mla_out_proj_fused_workspace_bytes": (_SZ, [_I, _I, _I]),
    "mla_out_proj_fused": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "mla_prefill_workspace_bytes": (_SZ, [_I, _I64, _I]),
    "mla_copy_from_host": (_I, [_P, _P, _SZ, _P]),
    "mla_prefill": (_I, [_P, _P, _P, _I64, _I, _P, _P, _I, _I, _I, _F, _P, _P, _P, _SZ, _P, _P]),
}

_LIB = None


class MLAError(RuntimeError):
    def __init__(self, call: str, code: int):
        super().__init__(f"{call} returned {STATUS.get(code, code)}")
        self.code = code


def lib() -> ctypes.CDLL:
    """The loaded libmla.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m mla_latent_kv_70_b300.build` (nvcc, sm_103a)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype, fn.argtypes = res, args
        _LIB = handle
    return _LIB


_BF16, _F32, _I32, _U8 = torch.bfloat16, torch.float32, torch.int32, torch.uint8


def _ptr(t, dtype=None):
    """Device address of tensor `t` (None -> NULL; an int passes through as an address).
    The library reads each buffer with the element type its header states, so a tensor of
    another dtype is refused here rather than misread."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"libmla expects a {dtype} tensor here, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError("libmla takes device tensors")
    if not t.is_contiguous():
        raise ValueError("libmla takes contiguous tensors")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(name, code):
    if code != 0:
        raise MLAError(name, code)


def mla_status_string(code: int) -> str:
    return lib().mla_status_string(code).decode()


def mla_device_sm_count() -> int:
    return lib().mla_device_sm_count()


def mla_absorb_q(q_nope, q_rope, w_uk, q_pos, rope_theta, q_cat, stream=None):
    """q_cat[b,s,h] = [q_nope[b,s,h] . W_UK[h]^T | RoPE(q_rope[b,s,h], q_pos[b,s])]."""
    B, S, H, _ = q_nope.shape
    _check("mla_absorb_q", lib().mla_absorb_q(
        _ptr(q_nope, _BF16), _ptr(q_rope, _BF16), _ptr(w_uk, _BF16), _ptr(q_pos, _I32),
        float(rope_theta), B, S, H, _ptr(q_cat, _BF16), _stream(stream)))


def mla_decode_workspace_bytes(B, S, H, num_splits, max_seqlen) -> int:
    return int(lib().mla_decode_workspace_bytes(B, S, H, num_splits, max_seqlen))


def mla_decode_num_splits(B, S, H, max_seqlen, total_rows=0) -> int:
    return int(lib().mla_decode_num_splits(B, S, H, max_seqlen, int(total_rows)))


def mla_decode_plan_splits(seqlens, S, H, *, causal=False, max_seqlen=None) -> int:
    """Split count from the batch's host-side lengths (a list or CPU int tensor)."""
    import ctypes
    lens = [int(x) for x in (seqlens.tolist() if hasattr(seqlens, "tolist") else seqlens)]
    if not lens:
        raise ValueError("empty batch")
    arr = (ctypes.c_int32 * len(lens))(*lens)
    T = max(lens) if max_seqlen is None else int(max_seqlen)
    r = int(lib().mla_decode_plan_splits(ctypes.addressof(arr), len(lens), int(S), int(H), 1 if causal else 0, T))
    if r < 1:
        raise ValueError("mla_decode_plan_splits rejected its arguments")
    return r


def mla_decode_latent(q_cat, kv, seqlens, o_lat, lse, *, scale, max_seqlen, block_table=None,
                      kv_seq_stride=0, page_size=64, causal=False, num_splits=0,
                      workspace=None, status=None, stream=None):
    """Absorbed attention over the latent cache; writes o_lat [B,S,H,512] and lse [B,S,H]."""
    B, S, H, _ = q_cat.shape
    if block_table is not None:
        num_pages, max_pages = kv.shape[0], block_table.shape[1]
    else:
        num_pages, max_pages = 0, 0
        kv_seq_stride = kv_seq_stride or kv.shape[1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("mla_decode_latent", lib().mla_decode_latent(
        _ptr(q_cat, _BF16), _ptr(kv, _BF16), int(kv_seq_stride), _ptr(seqlens, _I32),
        _ptr(block_table, _I32), max_pages, page_size, num_pages, B, S, H, int(bool(causal)),
        float(scale), int(num_splits), int(max_seqlen), _ptr(o_lat, _F32), _ptr(lse, _F32),
        _ptr(workspace), ws_bytes, _ptr(status, _I32), _stream(stream)))


def mla_quantize_fp8(rows, kv8, kv_scale, *, stream=None):
    """bf16 cache rows [n, 576] (rows may be a view with a larger row stride) -> the FP8
    form: kv8 uint8 [n, 640], kv_scale fp32 [n]."""
    if rows.dtype != _BF16 or not rows.is_cuda or rows.dim() != 2 or rows.shape[1] != 576 or rows.stride(1) != 1:
        raise ValueError("rows: a CUDA bf16 [n, 576] tensor with unit column stride")
    n = rows.shape[0]
    if kv8.numel() < n * 640 or kv_scale.numel() < n:
        raise ValueError("output too small")
    _check("mla_quantize_fp8", lib().mla_quantize_fp8(rows.data_ptr(), int(rows.stride(0)), n, _ptr(kv8, _U8),
                                                      _ptr(kv_scale, _F32), _stream(stream)))


def mla_append_latent_fp8(rows, seqlens, kv8, kv_scale, *, rope_theta=0.0, block_table=None, kv_seq_stride=0,
                          page_size=64, status=None, stream=None):
    """mla_append_latent into the FP8 form of the cache (kv8 uint8 [..., 640], kv_scale fp32)."""
    B, S, _ = rows.shape
    if block_table is not None:
        num_pages, max_pages = kv8.shape[0], block_table.shape[1]
    else:
        num_pages, max_pages = 0, 0
        kv_seq_stride = kv_seq_stride or kv8.shape[1]
    _check("mla_append_latent_fp8", lib().mla_append_latent_fp8(
        _ptr(rows, _BF16), B, S, float(rope_theta), _ptr(seqlens, _I32), _ptr(kv8, _U8), _ptr(kv_scale, _F32),
        int(kv_seq_stride), _ptr(block_table, _I32), max_pages, page_size, num_pages,
        _ptr(status, _I32), _stream(stream)))


def mla_decode_latent_fp8(q_cat, kv8, kv_scale, seqlens, o_lat, lse, *, scale, max_seqlen,
                          block_table=None, kv_seq_stride=0, page_size=64, causal=False,
                          num_splits=0, workspace=None, status=None, stream=None):
    """mla_decode_latent over the FP8 form of the cache (kv8 uint8 [..., 640], kv_scale fp32)."""
    B, S, H, _ = q_cat.shape
    if block_table is not None:
        num_pages, max_pages = kv8.shape[0], block_table.shape[1]
    else:
        num_pages, max_pages = 0, 0
        kv_seq_stride = kv_seq_stride or kv8.shape[1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("mla_decode_latent_fp8", lib().mla_decode_latent_fp8(
        _ptr(q_cat, _BF16), _ptr(kv8, _U8), _ptr(kv_scale, _F32), int(kv_seq_stride), _ptr(seqlens, _I32),
        _ptr(block_table, _I32), max_pages, page_size, num_pages, B, S, H, int(bool(causal)),
        float(scale), int(num_splits), int(max_seqlen), _ptr(o_lat, _F32), _ptr(lse, _F32),
        _ptr(workspace), ws_bytes, _ptr(status, _I32), _stream(stream)))


def mla_decode_latent_noalloc(q_cat, kv, seqlens, o_lat, lse, *, scale, max_seqlen,
                              block_table=None, kv_seq_stride=0, page_size=64, causal=False,
                              num_splits=0, status=None, stream=None):
    """mla_decode_latent with the split partials in the library's fixed scratch array
    (for callers that cannot allocate device memory); see include/mla.h."""
    B, S, H, _ = q_cat.shape
    if block_table is not None:
        num_pages, max_pages = kv.shape[0], block_table.shape[1]
    else:
        num_pages, max_pages = 0, 0
        kv_seq_stride = kv_seq_stride or kv.shape[1]
    _check("mla_decode_latent_noalloc", lib().mla_decode_latent_noalloc(
        _ptr(q_cat, _BF16), _ptr(kv, _BF16), int(kv_seq_stride), _ptr(seqlens, _I32),
        _ptr(block_table, _I32), max_pages, page_size, num_pages, B, S, H, int(bool(causal)),
        float(scale), int(num_splits), int(max_seqlen), _ptr(o_lat, _F32), _ptr(lse, _F32),
        _ptr(status, _I32), _stream(stream)))


def mla_combine_partials(o_part, lse_part, o_lat, lse, stream=None):
    splits = o_part.shape[0]
    rows = lse_part.numel() // splits
    _check("mla_combine_partials", lib().mla_combine_partials(
        _ptr(o_part, _F32), _ptr(lse_part, _F32), splits, rows, _ptr(o_lat, _F32), _ptr(lse, _F32),
        _stream(stream)))


def mla_out_proj_uv(o_lat, w_uv, o, stream=None):
    B, S, H, _ = o_lat.shape
    _check("mla_out_proj_uv", lib().mla_out_proj_uv(_ptr(o_lat, _F32), _ptr(w_uv, _BF16), B, S, H,
                                                    _ptr(o, _F32), _stream(stream)))


def mla_append_latent(rows, seqlens, kv, *, rope_theta=0.0, block_table=None, kv_seq_stride=0,
                      page_size=64, status=None, stream=None):
    """Write rows [B,S,576] at positions seqlens[b] + s of the cache (k^R rotated when
    rope_theta > 0) and advance seqlens by S."""
    B, S, _ = rows.shape
    if block_table is not None:
        num_pages, max_pages = kv.shape[0], block_table.shape[1]
    else:
        num_pages, max_pages = 0, 0
        kv_seq_stride = kv_seq_stride or kv.shape[1]
    _check("mla_append_latent", lib().mla_append_latent(
        _ptr(rows, _BF16), B, S, float(rope_theta), _ptr(seqlens, _I32), _ptr(kv, _BF16),
        int(kv_seq_stride), _ptr(block_table, _I32), max_pages, page_size, num_pages,
        _ptr(status, _I32), _stream(stream)))


def mla_fuse_weights(w_uq, w_uk, w_uv, w_o, w_uqk, w_uvo, stream=None):
    """W_UQK[h] = W_UQ[h] W_UK[h]^T and W_UVO[h] = W_UV[h] W_O[h] (bf16 outputs)."""
    H, d_cq, _ = w_uq.shape
    d_model = w_o.shape[2]
    _check("mla_fuse_weights", lib().mla_fuse_weights(
        _ptr(w_uq, _BF16), _ptr(w_uk, _BF16), _ptr(w_uv, _BF16), _ptr(w_o, _BF16), H, d_cq, d_model,
        _ptr(w_uqk, _BF16), _ptr(w_uvo, _BF16), _stream(stream)))


def mla_absorb_q_fused(c_q, q_rope, w_uqk, q_pos, rope_theta, q_cat, stream=None):
    """q_cat[b,s,h] = [c_q[b,s] . W_UQK[h] | RoPE(q_rope[b,s,h], q_pos[b,s])]."""
    B, S, H, _ = q_rope.shape
    d_cq = c_q.shape[2]
    _check("mla_absorb_q_fused", lib().mla_absorb_q_fused(
        _ptr(c_q, _BF16), _ptr(q_rope, _BF16), _ptr(w_uqk, _BF16), _ptr(q_pos, _I32), float(rope_theta),
        B, S, H, d_cq, _ptr(q_cat, _BF16), _stream(stream)))


def mla_out_proj_fused_workspace_bytes(B, S, H) -> int:
    return int(lib().mla_out_proj_fused_workspace_bytes(B, S, H))


def mla_out_proj_fused(o_lat, w_uvo, out, workspace, stream=None):
    """out[b,s] = sum_h o_lat[b,s,h] . W_UVO[h] (fp32)."""
    B, S, H, _ = o_lat.shape
    d_model = w_uvo.shape[2]
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("mla_out_proj_fused", lib().mla_out_proj_fused(
        _ptr(o_lat, _F32), _ptr(w_uvo, _BF16), B, S, H, d_model, _ptr(out, _F32), _ptr(workspace),
        ws_bytes, _stream(stream)))


def mla_prefill_workspace_bytes(B, kv_seq_stride, H) -> int:
    return int(lib().mla_prefill_workspace_bytes(B, int(kv_seq_stride), H))


def mla_prefill(q_nope, q_rope, kv, T_kv, w_uk, w_uv, o, lse, *, scale, workspace, status=None,
                stream=None):
    """Causal attention of the T_q query tokens (the last T_q of T_kv positions) of each
    sequence over expanded per-head keys/values; writes o [B,T_q,H,128] and lse [B,T_q,H]."""
    B, T_q, H, _ = q_nope.shape
    stride = kv.shape[1]
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("mla_prefill", lib().mla_prefill(
        _ptr(q_nope, _BF16), _ptr(q_rope, _BF16), _ptr(kv, _BF16), int(stride), int(T_kv), _ptr(w_uk, _BF16),
        _ptr(w_uv, _BF16), B, T_q, H, float(scale), _ptr(o, _F32), _ptr(lse, _F32), _ptr(workspace), ws_bytes,
        _ptr(status, _I32), _stream(stream)))


def mla_copy_from_host(dst, src_pinned, stream=None):
    """dst (device) <- src_pinned (pinned host tensor of the same size), copied by the SMs."""
    if src_pinned.is_cuda or not src_pinned.is_pinned():
        raise ValueError("mla_copy_from_host takes a pinned host tensor")
    nbytes = src_pinned.numel() * src_pinned.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("size mismatch")
    _check("mla_copy_from_host", lib().mla_copy_from_host(_ptr(dst), src_pinned.data_ptr(), nbytes,
                                                          _stream(stream)))


def mla_rope_inplace(x, row_stride, rows, col_offset, pos, theta, stream=None):
    _check("mla_rope_inplace", lib().mla_rope_inplace(_ptr(x, _BF16), int(row_stride), int(rows),
                                                      int(col_offset), _ptr(pos, _I32), float(theta),
                                                      _stream(stream)))


FAULT_DECODE, FAULT_ABSORB, FAULT_OUT_PROJ = 1, 2, 4


def mla_debug_inject_timeout(kernels: int, wait_ms: float = 1.0) -> None:
    """Test hook: the named kernels shorten their waits to `wait_ms` and withhold one
    completion signal, so that a bounded wait runs out (0 turns it off); see mla.h."""
    _check("mla_debug_inject_timeout", lib().mla_debug_inject_timeout(int(kernels), float(wait_ms)))


from .pipeline import DecodeStep  # noqa: E402,F401
