"""The layer call's bounded waits, made to run out on purpose without any
fault: a test hook shortens the bound on waits for other blocks' exchange
words to a few cycles, so the launch gives up, records MOE_DEV_TIMEOUT in the
status word, skips the rest of its work and returns with the context intact.
After the bound is restored and the workspace zero-filled (the recovery the
header prescribes), the next call is correct again."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_y_close

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("quantized_routed_expert_router_gb300")
from quantized_routed_expert_router_gb300.device_layer import DeviceLayer  # noqa: E402


@pytest.mark.parametrize("T", [1, 3])
def test_exchange_wait_timeout_then_recovery(T):
    cfg = synth.shrink(synth.CONFIGS["a3b"], H=1024, I=512, E=16, k=4, shared_I=256)
    L = synth.make_layer(cfg, 0, T=T)
    ref = oracle.layer_forward(L)
    dl = DeviceLayer(L, "cuda")
    try:
        moe.moe_debug_set_exchange_wait(50)
        dl.forward_fused(outputs=False)
        torch.cuda.synchronize()
        flags = moe.moe_read_device_status(dl.ws_layer, clear=False)
        assert flags & moe.DEV_TIMEOUT, flags
    finally:
        moe.moe_debug_set_exchange_wait(0)
    torch.cuda.synchronize()                  # the context is still usable
    dl.ws_layer.zero_()
    for _ in range(2):
        dl.y.fill_(float("nan"))
        dl.forward_fused()
        torch.cuda.synchronize()
        assert moe.moe_read_device_status(dl.ws_layer) == 0
        assert np.array_equal(dl.ids.cpu().numpy(), ref["ids"])
        assert_y_close(dl.y.cpu().numpy(), ref["y"], "after recovery")


def test_exchange_wait_hook_rejects_negative_bounds():
    with pytest.raises(moe.MoeError):
        moe.moe_debug_set_exchange_wait(-1)
