"""Stream and CUDA-graph behaviour of the C-ABI calls.

Every libmsda call only enqueues kernels on the stream it is given, so it
must (1) honour a non-default stream, (2) give the same results when two
problems run concurrently on two streams, and (3) replay correctly from a
captured CUDA graph (forward + backward with a caller-provided workspace)."""
import numpy as np
import pytest
import torch

from scale_deformable_attention_msda_gb300 import binding, workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _inputs(w, dt=torch.bfloat16):
    p = wl.make_inputs(w)
    t = {k: torch.tensor(p[k], dtype=torch.float64).to(dt).cuda()
         for k in ("value", "loc", "attn", "grad_out")}
    t["shapes"] = torch.tensor(p["shapes"]).cuda()
    t["starts"] = torch.tensor(p["starts"]).cuda()
    return t


def _run(t, stream=None, buf=None):
    out = binding.msda_forward(t["value"], t["shapes"], t["starts"], t["loc"], t["attn"],
                               stream=stream)
    kw = {}
    if buf is not None:
        kw = dict(grad_value=buf.grad_value, grad_sampling_locations=buf.grad_sampling_locations,
                  grad_attention_weights=buf.grad_attention_weights, workspace=buf.workspace,
                  accum=buf.accum)
    gv, gl, ga = binding.msda_backward(t["value"], t["shapes"], t["starts"], t["loc"], t["attn"],
                                       t["grad_out"], stream=stream, **kw)
    return out, gv, gl, ga


def _close(a, b, tol=2e-2):
    a, b = a.double(), b.double()
    return float((a - b).norm() / max(b.norm().item(), 1e-30)) <= tol


def test_non_default_stream():
    t = _inputs(wl.decoder("bf16"))
    ref = [x.clone() for x in _run(t)]
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        got = _run(t, stream=s)
    s.synchronize()
    assert torch.equal(got[0], ref[0]) and torch.equal(got[2], ref[2]) and torch.equal(got[3], ref[3])
    assert _close(got[1], ref[1])


def test_two_streams_concurrently():
    a, b = _inputs(wl.decoder("bf16")), _inputs(wl.sweep(5000, 4, 4))
    ra, rb = [x.clone() for x in _run(a)], [x.clone() for x in _run(b)]
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(s1):
        ga = _run(a, stream=s1)
    with torch.cuda.stream(s2):
        gb = _run(b, stream=s2)
    torch.cuda.synchronize()
    for got, ref in ((ga, ra), (gb, rb)):
        assert torch.equal(got[0], ref[0]) and torch.equal(got[2], ref[2])
        assert _close(got[1], ref[1])


def test_cuda_graph_capture_and_replay():
    t = _inputs(wl.encoder("bf16"))
    buf = binding.BackwardBuffers(t["value"], t["loc"], t["attn"], binding.MSDA_ACC_FP32_BUFFER)
    eager = [x.clone() for x in _run(t, buf=buf)]
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):               # warm up outside the capture
        _run(t, stream=s, buf=buf)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        outs = _run(t, stream=torch.cuda.current_stream(), buf=buf)
    for _ in range(3):
        buf.grad_value.fill_(7.0)             # the replay must overwrite everything
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(outs[0], eager[0]) and torch.equal(outs[2], eager[2])
    assert torch.equal(outs[3], eager[3])
    assert _close(outs[1], eager[1])
    # new inputs copied into the captured buffers are picked up by the replay
    t2 = _inputs(wl.encoder("bf16", variant=1))
    for k in ("value", "loc", "attn", "grad_out"):
        t[k].copy_(t2[k])
    g.replay()
    fresh = _run(t2)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], fresh[0]) and torch.equal(outs[2], fresh[2])


def test_cuda_graph_with_auto_accumulation():
    """MSDA_ACC_AUTO is resolved on the host, so a captured call replays the
    mode it resolved to: on the decoder shape native adds with no workspace,
    zeroing grad_value on every replay."""
    t = _inputs(wl.decoder("bf16"))
    buf = binding.BackwardBuffers(t["value"], t["loc"], t["attn"], binding.MSDA_ACC_AUTO)
    assert buf.workspace is None                    # resolved to native: nothing to allocate
    eager = [x.clone() for x in _run(t, buf=buf)]
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _run(t, stream=s, buf=buf)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        outs = _run(t, stream=torch.cuda.current_stream(), buf=buf)
    for _ in range(3):
        buf.grad_value.fill_(7.0)
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(outs[0], eager[0]) and torch.equal(outs[2], eager[2])
    assert torch.equal(outs[3], eager[3])
    assert _close(outs[1], eager[1])


def test_cuda_graph_with_fp16_buffer_rescales_every_replay():
    """MSDA_ACC_FP16_BUFFER derives its scale on the device from the
    current grad_out and attention weights, so a captured call must follow
    new inputs: grad_out 1000 times larger copied into the captured buffer
    gives a grad_value 1000 times larger, not an overflowed one."""
    t = _inputs(wl.encoder("bf16"))
    buf = binding.BackwardBuffers(t["value"], t["loc"], t["attn"], binding.MSDA_ACC_FP16_BUFFER)
    assert buf.workspace is not None
    eager = [x.clone() for x in _run(t, buf=buf)]
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _run(t, stream=s, buf=buf)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        outs = _run(t, stream=torch.cuda.current_stream(), buf=buf)
    for _ in range(3):
        buf.grad_value.fill_(7.0)
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(outs[2], eager[2]) and torch.equal(outs[3], eager[3])
    assert _close(outs[1], eager[1], tol=1e-2)      # the adds' order varies between runs
    t["grad_out"].mul_(1000.0)                       # exact in bf16 up to rounding of x1000
    fresh_buf = binding.BackwardBuffers(t["value"], t["loc"], t["attn"],
                                        binding.MSDA_ACC_FP16_BUFFER)
    fresh = _run(t, buf=fresh_buf)
    g.replay()
    torch.cuda.synchronize()
    assert torch.isfinite(outs[1].float()).all()
    assert _close(outs[1], fresh[1], tol=1e-2)
    assert _close(outs[1], eager[1].double() * 1000.0, tol=2e-2)


def test_fp16_buffer_on_two_streams():
    """Two problems with their own fp16 workspaces on two streams at once."""
    a, b = _inputs(wl.encoder("bf16")), _inputs(wl.sweep(5000, 4, 4, contention=True))
    bufs = [binding.BackwardBuffers(x["value"], x["loc"], x["attn"], binding.MSDA_ACC_FP16_BUFFER)
            for x in (a, b)]
    ra, rb = [x.clone() for x in _run(a, buf=bufs[0])], [x.clone() for x in _run(b, buf=bufs[1])]
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    bufs2 = [binding.BackwardBuffers(x["value"], x["loc"], x["attn"], binding.MSDA_ACC_FP16_BUFFER)
             for x in (a, b)]
    with torch.cuda.stream(s1):
        ga = _run(a, stream=s1, buf=bufs2[0])
    with torch.cuda.stream(s2):
        gb = _run(b, stream=s2, buf=bufs2[1])
    torch.cuda.synchronize()
    for got, ref in ((ga, ra), (gb, rb)):
        assert torch.equal(got[0], ref[0]) and torch.equal(got[2], ref[2])
        assert torch.equal(got[3], ref[3])
        assert _close(got[1], ref[1], tol=1e-2)


def test_calls_from_two_host_threads():
    """Two host threads, each with its own stream and buffers, issue forward
    and backward calls at the same time (ctypes releases the GIL during the
    calls); every result matches the same calls made from one thread. The
    range-checked library runs the same way, so its per-context fault-word
    lookup is taken from both threads at once."""
    import threading

    from scale_deformable_attention_msda_gb300 import build
    problems = [_inputs(wl.decoder("bf16")), _inputs(wl.sweep(5000, 4, 4))]
    refs = [[x.clone() for x in _run(t)] for t in problems]
    torch.cuda.synchronize()
    for lib in (build.LIBRARY, build.CHECKED_LIBRARY):
        binding.use_library(lib)
        try:
            results, errors = [None, None], []

            def work(i):
                try:
                    s = torch.cuda.Stream()
                    with torch.cuda.stream(s):
                        for _ in range(10):
                            got = _run(problems[i], stream=s)
                    s.synchronize()
                    results[i] = got
                except Exception as e:                # reported on the main thread
                    errors.append(e)

            threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
            for th in threads:
                th.start()
            for th in threads:
                th.join()
            assert not errors, errors
            torch.cuda.synchronize()
            assert binding.msda_device_check() == 0
            for got, ref in zip(results, refs):
                assert torch.equal(got[0], ref[0]) and torch.equal(got[2], ref[2])
                assert torch.equal(got[3], ref[3])
                assert _close(got[1], ref[1])
        finally:
            binding.use_library(build.LIBRARY)
