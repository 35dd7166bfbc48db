"""Decode-sized forwards from two host threads at once.  Their shared experts run on a stream the
library forks per call; that stream belongs to the calling thread, so two threads never queue
behind each other there, and one thread's stream capture does not pull in the other thread's
shared-expert work.  Every output must equal the single-threaded bytes."""
import threading

import pytest
import torch

import moe_synth
from sparse_conditional_moe_b300 import moe

from gpu_util import to_dev

pytestmark = pytest.mark.gpu

SPEC = moe_synth.LayerSpec("decode_threads", N=64, d=512, d_ff=256, E=32, k=4, n_shared=1,
                           d_ff_shared=256)


def _layers():
    out = []
    for seed in (3, 4):
        dev = to_dev(moe_synth.make_layer(SPEC, seed=seed))
        lay = moe.MoELayer(moe.cfg_from_spec(SPEC), dev)
        ref = lay.forward(dev["x"]).clone()
        out.append((lay, dev, ref))
    torch.cuda.synchronize()
    return out


def _run_threads(targets):
    errors = []

    def wrap(fn):
        def go():
            try:
                torch.cuda.set_device(0)
                fn()
            except BaseException as e:   # noqa: BLE001 -- reported below
                errors.append(e)
        return go

    ts = [threading.Thread(target=wrap(t)) for t in targets]
    for t in ts:
        t.start()
    for t in ts:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in ts), "a thread did not finish"
    assert not errors, errors


def test_two_threads_forward_concurrently():
    layers = _layers()

    def worker(i):
        def run():
            lay, dev, ref = layers[i]
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                for _ in range(40):
                    out = lay.forward(dev["x"], stream=st)
                st.synchronize()
                assert torch.equal(out, ref)
                assert lay.device_error(st) == 0
        return run

    _run_threads([worker(0), worker(1)])


def test_capture_in_one_thread_while_another_runs_eagerly():
    layers = _layers()
    graph = {}
    started = threading.Event()

    def capture():
        lay, dev, ref = layers[0]
        x = dev["x"].clone()
        st = torch.cuda.Stream()
        with torch.cuda.stream(st):
            lay.forward(x, stream=st)           # this thread's side stream exists before capture
            st.synchronize()
            started.wait(timeout=60)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st, capture_error_mode="thread_local"):
                lay.forward(x, stream=st)
            st.synchronize()
        graph["g"], graph["x"] = g, x

    def eager():
        lay, dev, ref = layers[1]
        st = torch.cuda.Stream()
        with torch.cuda.stream(st):
            started.set()
            for _ in range(60):
                out = lay.forward(dev["x"], stream=st)
            st.synchronize()
            assert torch.equal(out, ref)

    _run_threads([capture, eager])
    lay, dev, ref = layers[0]
    lay.out.zero_()
    graph["g"].replay()
    torch.cuda.synchronize()
    assert lay.device_error() == 0
    assert torch.equal(lay.out, ref)
