"""One cycle through spec_cycle_host: the step's inputs start in page-locked
host memory, the library copies them in, drafts, verifies and copies the
results back.  The host results must match the float64 oracle exactly as
the device-resident cycle does, with the target copy on a second stream and
without, and the device buffers the call filled must hold the host inputs."""
import numpy as np
import pytest

from speculative_decoding_draft_04_gb300 import workloads as W

from parity import GpuResult, assert_parity, compare, oracle_cycle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = pytest.importorskip("torch")
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_draft_04_gb300 import build as B
    B.build()
    return t


def host_cycle(torch, w, copy_stream):
    from speculative_decoding_draft_04_gb300 import engine
    d = engine.DeviceWorkload.from_workload(w)
    h = engine.HostStep.like(d)
    # the device input buffers start out holding something else
    for t in (d.U, d.target, d.verify_len):
        t.zero_()
    d.anchor.fill_(1)
    for t in (d.temperature, d.u_draft, d.u_accept, d.u_final):
        t.fill_(0.5)
    b = engine.Buffers.for_workload(d)
    cs = torch.cuda.Stream() if copy_stream else None
    engine.cycle_host(d, b, h, copy_stream=cs, extras=True)
    torch.cuda.synchronize()
    for k in ("U", "target", "anchor", "temperature", "u_draft", "verify_len", "u_accept",
              "u_final"):
        assert torch.equal(getattr(d, k).cpu(), getattr(h, k)), k
    g = GpuResult(h.draft_tokens.numpy(), b.q_tok.cpu().numpy(), b.lse_q.cpu().numpy(),
                  h.accept_len.numpy(), h.out_tokens.numpy(), h.alpha.numpy(),
                  b.p_tok.cpu().numpy(), engine.status_words(b.dstatus),
                  engine.status_words(b.vstatus), None, None)
    assert np.array_equal(g.draft_tokens, b.draft_tokens.cpu().numpy())
    assert np.array_equal(g.out_tokens, b.out_tokens.cpu().numpy())
    return g


@pytest.mark.parametrize("copy_stream", [False, True])
@pytest.mark.parametrize("name,B", [("C0", None), ("C4", 24)])
def test_host_cycle_matches_the_oracle(torch, name, B, copy_stream):
    w = W.make_workload(W.config(name), trial=3, B=B)
    g = host_cycle(torch, w, copy_stream)
    assert_parity(compare(w, g, oracle_cycle(w)))
