"""The forward pass under CUDA-graph capture: a captured moe_forward replays to the same bytes
as the eager call.  This covers the decode path that forks the shared experts onto the
library's own stream (the fork and join become graph edges), the W4A16 forward, layers with
capacity dropping, the tensor-core router's cluster launch and the permutation's cooperative
launch.  No launch inside the forward allocates, synchronises or reads back, which is
what capture requires."""
import pytest
import torch

import moe_synth
from sparse_conditional_moe_b300 import moe

from gpu_util import to_dev

pytestmark = pytest.mark.gpu

CASES = [
    moe_synth.LayerSpec("decode_shared", N=64, d=512, d_ff=256, E=32, k=4, n_shared=1,
                        d_ff_shared=256),
    moe_synth.LayerSpec("prefill_capacity", N=640, d=256, d_ff=384, E=16, k=2, n_shared=1,
                        d_ff_shared=128, capacity_factor=1.0),
    moe_synth.LayerSpec("decode_w4", N=32, d=512, d_ff=256, E=16, k=4, n_shared=1,
                        d_ff_shared=256, w4a16=True),
    # the tensor-core router in its fused cluster form (E = 256, batch over 1024 tokens) and in
    # its unfused form with the top-k kernel (E = 128); every case groups its assignments with
    # the cooperative permutation kernel
    moe_synth.LayerSpec("fused_router", N=1100, d=512, d_ff=256, E=256, k=8, n_shared=1,
                        d_ff_shared=256),
    moe_synth.LayerSpec("tc_router_capacity", N=2048, d=512, d_ff=256, E=128, k=4,
                        capacity_factor=1.25, zipf_bias=1.2),
]


@pytest.mark.parametrize("spec", CASES, ids=lambda s: s.name)
def test_captured_forward_replays_to_the_eager_bytes(spec):
    dev = to_dev(moe_synth.make_layer(spec, seed=9))
    w4 = moe.quantize_layer_w4(dev) if spec.w4a16 else None
    lay = moe.MoELayer(moe.cfg_from_spec(spec), dev, w4=w4)
    x = dev["x"].clone()
    eager = lay.forward(x).clone()              # also creates the library's side stream
    torch.cuda.synchronize()
    g = lay.capture(x)
    lay.out.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert lay.device_error() == 0
    assert torch.equal(lay.out, eager)
    # a new input in the captured buffer flows through the replay
    x.copy_(torch.flip(dev["x"], [0]))
    g.replay()
    torch.cuda.synchronize()
    want = lay.forward(x.clone()).clone()
    torch.cuda.synchronize()
    assert torch.equal(want, lay.out)
