"""The bounded device-side waits: when a wait runs out, the kernel records a timeout in
the status word and returns (no trap, no hang), the host reads the status, and the
context stays usable.  The waits are made to run out by setting their poll budget to
one poll through the test hook; nothing is broken on the device."""
import numpy as np
import pytest

import workloads as W
from helpers import check_case, ensure_built, upload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", [
    W.Case(1, 8, 2, 512, 2048, 128, 128, "bf16", "causal", False, None, "n0.5", seed=21,
           name="prefill_tc"),
    W.Case(4, 32, 4, 1, 20000, 128, 128, "f16", "causal", True, None, "u2", seed=22,
           name="decode_mma"),
], ids=lambda c: c.name)
def test_wait_timeout_is_reported_and_context_survives(case):
    import torch
    nv = ensure_built()
    x = W.make_inputs(case)
    dev = upload(case, x)
    assert nv.nv_sdpa_device_status(0) == (nv.OK, 0)
    try:
        nv.nv_sdpa_set_wait_limit(1)
        nv.sdpa(dev["q"], dev["k"], dev["v"], mask_kind=case.mask, scale=case.scale_f32,
                sinks=dev["sinks"])
        st, detail = nv.nv_sdpa_device_status(0)
    finally:
        nv.nv_sdpa_set_wait_limit(0)
    assert st == nv.ERR_DEVICE_TIMEOUT and detail != 0, (st, detail)
    # the status word was cleared by the read, and the next call is correct
    assert nv.nv_sdpa_device_status(0) == (nv.OK, 0)
    check_case(case, x, max_oracle_flops=1e12)
    torch.cuda.synchronize()
