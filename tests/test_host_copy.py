"""mla_copy_from_host: the SM-driven copy out of pinned host memory that the serving loop in
bench.py uses for its queries.  It is no step of the method, so the check is a plain one:
the bytes arrive unchanged, at sizes that leave a partial last round of the grid-stride
loop, and the call refuses what it cannot copy (null, unaligned or odd-sized buffers on
the host; pageable host memory, found by the runtime)."""
import ctypes

import pytest
import torch

import mla_latent_kv_70_b300 as mla
from mla_latent_kv_70_b300 import build as mla_build

P = 4096  # a fake 16-byte aligned address: a call rejected on the host never dereferences it


@pytest.fixture(scope="module")
def lib():
    mla_build.build()
    return mla.lib()


@pytest.mark.parametrize("dst,src,nbytes", [
    (None, P, 64), (P, None, 64), (P, P, 40), (P + 8, P, 64), (P, P + 4, 64)])
def test_rejects_on_the_host(lib, dst, src, nbytes):
    assert lib.mla_copy_from_host(dst, src, nbytes, None) == 1


def test_zero_bytes_is_a_no_op(lib):
    assert lib.mla_copy_from_host(P, P, 0, None) == 0


@pytest.mark.gpu
@pytest.mark.parametrize("nbytes", [16, 4096 + 48, 3 << 20, (17 << 20) + 16 * 1001])
def test_copies_every_byte(lib, nbytes):
    g = torch.Generator().manual_seed(nbytes)
    src = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=g).pin_memory()
    dst = torch.zeros(nbytes + 64, dtype=torch.uint8, device="cuda")
    mla.mla_copy_from_host(dst[:nbytes], src)
    torch.cuda.synchronize()
    assert torch.equal(dst[:nbytes].cpu(), src)
    assert int(dst[nbytes:].count_nonzero()) == 0          # nothing written past the end


@pytest.mark.gpu
def test_refuses_pageable_memory(lib):
    src = torch.ones(4096, dtype=torch.uint8)                 # not pinned
    dst = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    code = lib.mla_copy_from_host(dst.data_ptr(), src.data_ptr(), 4096, None)
    assert code == 1
    with pytest.raises(ValueError):
        mla.mla_copy_from_host(dst, src)
