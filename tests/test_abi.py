"""The C ABI library loads, exports every symbol include/mla.h declares, and rejects bad
arguments on the host before touching the GPU (these tests need no GPU)."""
import ctypes
import os
import re

import pytest

import mla_latent_kv_70_b300 as mla
from mla_latent_kv_70_b300 import build as mla_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla.h")


@pytest.fixture(scope="module")
def lib():
    mla_build.build()
    return mla.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("mla_absorb_q", "mla_decode_latent", "mla_out_proj_uv",
                     "mla_decode_workspace_bytes", "mla_combine_partials", "mla_rope_inplace"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in mla.SIGNATURES, f"{name} has no binding"


def test_status_strings(lib):
    for code, name in mla.STATUS.items():
        assert mla.mla_status_string(code) == name
    assert mla.mla_status_string(99) == "MLA_ERR_UNKNOWN"


P = 4096  # a fake, 16-byte aligned "device" address: never dereferenced by a rejected call


def decode_args(**over):
    a = dict(q_cat=P, kv=P, kv_seq_stride=256, seqlens=P, block_table=None, max_pages=0,
             page_size=64, num_pages=0, B=4, S=1, H=16, causal=0, scale=0.07, num_splits=1,
             max_seqlen=256, o_lat=P, lse=P, workspace=None, workspace_bytes=0, status=None,
             stream=None)
    a.update(over)
    return list(a.values())


@pytest.mark.parametrize("over,code", [
    (dict(q_cat=None), 1), (dict(kv=None), 1), (dict(seqlens=None), 1), (dict(o_lat=None), 1),
    (dict(B=0), 1), (dict(H=12), 2), (dict(H=256), 2), (dict(S=5), 2), (dict(scale=0.0), 1),
    (dict(scale=float("nan")), 1), (dict(num_splits=129), 1), (dict(num_splits=-1), 1),
    (dict(kv_seq_stride=100), 1), (dict(q_cat=P + 2), 1),
    (dict(block_table=P, max_pages=4, page_size=32, num_pages=8), 2),
    (dict(block_table=P, max_pages=2, num_pages=8), 1),
    (dict(num_splits=4, max_seqlen=256), 4),
])
def test_decode_rejects_bad_arguments(lib, over, code):
    assert lib.mla_decode_latent(*decode_args(**over)) == code


def test_workspace_bytes(lib):
    assert lib.mla_decode_workspace_bytes(4, 1, 16, 1, 256) == 0
    assert lib.mla_decode_workspace_bytes(4, 1, 16, 3, 256) == 3 * 4 * 16 * 513 * 4
    assert lib.mla_decode_workspace_bytes(4, 1, 16, 129, 256) == 0


def test_other_calls_reject_bad_arguments(lib):
    assert lib.mla_absorb_q(None, P, P, None, 1e4, 4, 1, 16, P, None) == 1
    assert lib.mla_absorb_q(P, P, P, None, 1e4, 4, 1, 20, P, None) == 2
    assert lib.mla_absorb_q(P, P, P, P, 0.0, 4, 1, 16, P, None) == 1
    assert lib.mla_out_proj_uv(P, P, 4, 1, 0, P, None) == 1
    assert lib.mla_out_proj_uv(P, None, 4, 1, 16, P, None) == 1
    assert lib.mla_combine_partials(P, P, 0, 10, P, P, None) == 1
    assert lib.mla_combine_partials(P, P, 200, 10, P, P, None) == 1
    assert lib.mla_rope_inplace(P, 576, 10, 512, None, 1e4, None) == 1
    assert lib.mla_rope_inplace(P, 576, 10, 520, P, 1e4, None) == 1
    assert lib.mla_rope_inplace(P, 576, 10, 511, P, 1e4, None) == 1
    f = ctypes.c_float
    assert lib.mla_append_latent(None, 2, 1, f(1e4), P, P, 64, None, 0, 64, 0, None, None) == 1
    assert lib.mla_append_latent(P, 0, 1, f(1e4), P, P, 64, None, 0, 64, 0, None, None) == 1
    assert lib.mla_append_latent(P, 2, 1, f(-1.0), P, P, 64, None, 0, 64, 0, None, None) == 1
    assert lib.mla_append_latent(P + 8, 2, 1, f(1e4), P, P, 64, None, 0, 64, 0, None, None) == 1
    assert lib.mla_append_latent(P, 2, 1, f(1e4), P, P, 0, None, 0, 64, 0, None, None) == 1
    assert lib.mla_append_latent(P, 2, 1, f(1e4), P, P, 0, P, 4, 32, 10, None, None) == 2
    assert lib.mla_append_latent(P, 2, 1, f(1e4), P, P, 0, P, 0, 64, 10, None, None) == 1


# ----------------------------------------------------------------------------
# Split planner (host logic; without a GPU it assumes 148 SMs, as on a B300)
# ----------------------------------------------------------------------------

def test_planner_invariants(lib):
    for B, S, H, T in [(1, 1, 128, 1), (4, 1, 16, 256), (64, 1, 128, 4096), (2, 1, 128, 131072),
                       (128, 2, 128, 8192), (1, 1, 128, 10 ** 6), (300, 1, 128, 64)]:
        s = mla.mla_decode_num_splits(B, S, H, T)
        assert 1 <= s <= 128                      # MLA_MAX_SPLITS
        assert s <= -(-T // 64)                   # never more splits than 64-row tiles
    assert mla.mla_decode_num_splits(8, 1, 128, 0) == 1


@pytest.mark.parametrize("name,expected", [("tiny", 4), ("dsv3", 1), ("ragged_paged", 12),
                                           ("long_splitkv", 36), ("mtp", 2)])
def test_planner_choices_for_the_workloads(lib, name, expected):
    # The counts the measured results were taken with: a full machine of CTA pairs is
    # left unsplit; long or ragged batches are split to fill waves of 74 pairs.
    from mla_latent_kv_70_b300 import inputs as I
    c = getattr(I, name)()
    assert mla.mla_decode_num_splits(c.B, c.S, c.H, max(c.seqlens), c.total_tokens) == expected


def test_planner_uses_the_total_row_hint(lib):
    # Without the hint the planner assumes every sequence is max_seqlen long; a ragged
    # batch (about half that on average) fills fewer waves and is split more.
    from mla_latent_kv_70_b300 import inputs as I
    c = I.ragged_paged()
    T = max(c.seqlens)
    assert mla.mla_decode_num_splits(c.B, 1, 128, T, c.total_tokens) > mla.mla_decode_num_splits(c.B, 1, 128, T)


@pytest.mark.parametrize("name,expected", [("tiny", 1), ("dsv3", 1), ("ragged_paged", 8),
                                           ("long_splitkv", 36), ("mtp", 1)])
def test_length_planner_choices_for_the_workloads(lib, name, expected):
    # The counts that measured fastest on a B300 among those tried (ragged: 2-16, long
    # context: 24-48, multi-token: 1-3, DeepSeek-V3: 1-2; tiny: all equal).
    from mla_latent_kv_70_b300 import inputs as I
    c = getattr(I, name)()
    assert mla.mla_decode_plan_splits(c.seqlens, c.S, c.H, causal=c.causal) == expected


def _schedule_time(lens, S, H, causal, s, slots=74):
    """The planner's schedule estimate, restated: units in launch order, each to the pair
    slot that frees first; 17 us + 1.036 us per 64-row tile (11 us fixed for a unit
    starting after 3 us), 1.5 us for an empty unit, plus the merge for s > 1."""
    import heapq
    T = max(lens)
    chunk = ((T + s - 1) // s + 63) // 64 * 64
    free = [0.0] * slots
    for Tb in lens:
        for q in range(S):
            n_vis = min(Tb, max(0, Tb - S + q + 1)) if causal else Tb
            for k in range(s):
                t0 = min(k * chunk, n_vis)
                tiles = (min(t0 + chunk, n_vis) - t0 + 63) // 64
                t = heapq.heappop(free)
                heapq.heappush(free, t + ((17.0 if t < 3.0 else 11.0) + tiles * 1.036 if tiles else 1.5))
    t = max(free)
    if s > 1:
        t += 3.0 + s * len(lens) * S * H * 513 * 8 / 6.0e6
    return t


def test_length_planner_follows_its_schedule_model(lib):
    import random
    rng = random.Random(5)
    for trial in range(12):
        B = rng.choice([1, 3, 17, 64, 150])
        S = rng.choice([1, 2, 4])
        causal = S > 1 and rng.random() < 0.5
        lens = [rng.randint(0, 20000) for _ in range(B)]
        lens[0] = max(lens[0], 1)
        T = max(lens)
        times = {s: _schedule_time(lens, S, 128, causal, s) for s in range(1, min(128, (T + 63) // 64) + 1)}
        best, best_t = 1, times[1]
        for s in sorted(times)[1:]:
            if times[s] < best_t * 0.98:
                best, best_t = s, times[s]
        assert mla.mla_decode_plan_splits(lens, S, 128, causal=causal) == best, (B, S, causal)


def test_length_planner_edge_cases(lib):
    assert mla.mla_decode_plan_splits([0, 0, 0], 1, 128) == 1        # nothing readable
    assert mla.mla_decode_plan_splits([64] * 300, 1, 128) == 1       # one tile each
    for lens in ([1], [10 ** 6], [5, 10 ** 5, 7]):
        s = mla.mla_decode_plan_splits(lens, 1, 128)
        assert 1 <= s <= min(128, -(-max(lens) // 64))
    import ctypes
    arr = (ctypes.c_int32 * 2)(100, 200)
    f = lib.mla_decode_plan_splits
    assert f(None, 2, 1, 128, 0, 200) == 0                               # null lengths
    assert f(ctypes.addressof(arr), 0, 1, 128, 0, 200) == 0              # B < 1
    assert f(ctypes.addressof(arr), 2, 5, 128, 0, 200) == 0              # S > 4
    assert f(ctypes.addressof(arr), 2, 1, 24, 0, 200) == 0               # H not a multiple of 16
    assert f(ctypes.addressof(arr), 2, 1, 128, 0, 150) >= 1              # lengths clamped to max_seqlen


def test_binding_refuses_wrong_dtypes(lib):
    # The binding checks each tensor's element type (the library would misread it) before
    # its device; these CPU tensors stop at the first check that applies.
    import torch
    bf = lambda *s: torch.zeros(*s, dtype=torch.bfloat16)
    q32 = torch.zeros(2, 1, 16, 128, dtype=torch.float32)
    with pytest.raises(ValueError, match="bfloat16"):
        mla.mla_absorb_q(q32, bf(2, 1, 16, 64), bf(16, 512, 128), None, 1e4, bf(2, 1, 16, 576))
    with pytest.raises(ValueError, match="bfloat16"):
        mla.mla_decode_latent(torch.zeros(2, 1, 16, 576), bf(2, 64, 576), torch.zeros(2, dtype=torch.int32),
                              torch.zeros(2, 1, 16, 512), torch.zeros(2, 1, 16), scale=0.07, max_seqlen=64)
    with pytest.raises(ValueError, match="int32"):
        mla.mla_rope_inplace(17, 576, 1, 512, torch.zeros(1, dtype=torch.int64), 1e4)
    with pytest.raises(ValueError, match="float32"):
        mla.mla_out_proj_uv(bf(2, 1, 16, 512), bf(16, 512, 128), torch.zeros(2, 1, 16, 128))
    with pytest.raises(ValueError, match="device tensors"):   # right dtypes, host memory
        mla.mla_out_proj_uv(torch.zeros(2, 1, 16, 512), bf(16, 512, 128), torch.zeros(2, 1, 16, 128))


def test_timeout_hook_rejects_bad_arguments(lib):
    assert lib.mla_debug_inject_timeout(8, ctypes.c_double(1.0)) == 1        # unknown kernel bit
    assert lib.mla_debug_inject_timeout(1, ctypes.c_double(0.0)) == 1        # no wait limit
    assert lib.mla_debug_inject_timeout(1, ctypes.c_double(5000.0)) == 1     # beyond 2 s
    assert lib.mla_debug_inject_timeout(0, ctypes.c_double(0.0)) == 0        # off


def test_prefill_and_fused_calls_reject_bad_shapes(lib):
    f = ctypes.c_float

    def prefill(**kw):
        a = dict(qn=P, qr=P, kv=P, stride=128, T_kv=100, wuk=P, wuv=P, B=1, T_q=10, H=16, scale=f(0.07),
                 o=P, lse=P, ws=P, ws_bytes=1 << 30, status=None, stream=None)
        a.update(kw)
        return lib.mla_prefill(*a.values())
    assert prefill(T_q=200) == 1            # more query tokens than cached rows
    assert prefill(stride=50) == 1          # rows past the sequence stride
    assert prefill(H=24) == 2
    assert prefill(ws_bytes=16) == 4
    assert prefill(qn=P + 2) == 1
    assert lib.mla_fuse_weights(P, P, P, P, 16, 100, 4096, P, P, None) == 2          # d_cq % 64
    assert lib.mla_fuse_weights(P, P, P, P, 16, 1536, 1000, P, P, None) == 2         # d_model % 128
    assert lib.mla_absorb_q_fused(P, P, P, None, f(1e4), 2, 5, 16, 1536, P, None) == 2   # S > 4
    assert lib.mla_out_proj_fused(P, P, 2, 1, 16, 4096, P, P, 16, None) == 4          # workspace
