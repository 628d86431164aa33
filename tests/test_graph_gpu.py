"""The library's calls never synchronize or allocate, so a whole cycle
(memsets, the cooperative draft, the verification kernels) can be captured
into a CUDA graph; replaying it must give exactly the eager outputs."""
import numpy as np
import pytest

from speculative_decoding_draft_04_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_graph_replay_matches_eager():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_draft_04_gb300 import build, engine
    build.build()
    w = W.make_workload(W.config("C2"), trial=3, B=48)
    d = engine.DeviceWorkload.from_workload(w)
    b = engine.Buffers.for_workload(d)
    engine.cycle(d, b)
    torch.cuda.synchronize()
    eager = [t.clone() for t in (b.draft_tokens, b.q_tok, b.lse_q, b.accept_len, b.out_tokens, b.alpha)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        engine.cycle(d, b, side)
    for t in (b.draft_tokens, b.accept_len, b.out_tokens):
        t.fill_(-5)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for e, t in zip(eager, (b.draft_tokens, b.q_tok, b.lse_q, b.accept_len, b.out_tokens, b.alpha)):
        assert torch.equal(torch.nan_to_num(e, nan=-9.0), torch.nan_to_num(t, nan=-9.0))
    assert (engine.status_words(b.dstatus)[0] & ~16) == 0
