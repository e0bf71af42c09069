"""Device-side failure path: a bounded wait that runs out is reported, and the device
stays usable.

The test hook mla_debug_inject_timeout makes the chosen kernels withhold one completion
signal of their own and shortens their wait limit to 1 ms, so one of their waits runs out
(nothing is faulted: no trap, no bad address).  Each kernel must then record the timeout
(the decode) or write NaN (the projections), drain its copies and MMAs, free its tensor
memory and exit; the next ordinary step on the same device must match the oracle.
"""
import numpy as np
import pytest
import torch

from mla_latent_kv_70_b300 import inputs as I
from tests.mla_cases import DeviceCase, check_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_70_b300 import build
    build.build()


@pytest.fixture
def inject():
    import mla_latent_kv_70_b300 as mla
    yield mla.mla_debug_inject_timeout
    mla.mla_debug_inject_timeout(0)


@pytest.mark.parametrize("splits", [1, 3])
def test_decode_timeout_is_flagged_and_device_recovers(inject, splits):
    import mla_latent_kv_70_b300 as mla
    case = I.make_case("timeout", 3, 1, 128, [300, 130, 64], seed=61)
    dc = DeviceCase(case)
    inject(mla.FAULT_DECODE, 1.0)
    st = dc.step(num_splits=splits)
    assert int(st.status.item()) & mla.FLAG_TIMEOUT
    # Units that gave up write the empty result: o_lat = 0, lse = -inf (so o = 0).
    assert torch.all(st.o_lat == 0) and torch.all(torch.isneginf(st.lse))
    assert torch.all(st.o == 0)
    inject(0)
    st2 = dc.step(num_splits=splits)
    check_case(dc, st2, range(case.B))


def test_projection_timeouts_write_nan_and_device_recovers(inject):
    import mla_latent_kv_70_b300 as mla
    case = I.make_case("timeout_proj", 2, 1, 128, [200, 90], seed=63)
    dc = DeviceCase(case)
    inject(mla.FAULT_ABSORB, 1.0)
    st = dc.step(num_splits=1)
    q_cat = st.q_cat.float()
    assert torch.all(torch.isnan(q_cat[..., :512]))
    assert torch.equal(st.q_cat[..., 512:], dc.q_rope)        # the RoPE slice is still copied
    inject(mla.FAULT_OUT_PROJ, 1.0)
    st = dc.step(num_splits=1)
    assert int(st.status.item()) == 0                          # the decode itself ran normally
    assert torch.all(torch.isnan(st.o))
    assert torch.all(torch.isfinite(st.o_lat))
    inject(0)
    st = dc.step(num_splits=1)
    assert np.all(np.isfinite(st.o.cpu().numpy()))
    check_case(dc, st, range(case.B))
