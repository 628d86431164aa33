"""GPU parity of the tree path (spec_tree_select, spec_tree_draft,
spec_tree_verify) against the float64 tree oracle (oracle/tree.py): the
selected slots and survival values bit-exact, drafted tokens and the
verification's path, accept length and tokens bit-exact (both sides decide in
double precision; a mismatch is allowed only within 1e-9 of a boundary), q of
each drawn token within 1e-5."""
import numpy as np
import pytest

from oracle import tree as TR
from speculative_decoding_draft_04_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = pytest.importorskip("torch")
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_draft_04_gb300 import build as B
    B.build()
    return t


def _lib():
    from speculative_decoding_draft_04_gb300 import _lib as L
    return L


@pytest.mark.parametrize("B,N,gamma", [(1, 1, 1), (3, 9, 4), (64, 40, 7), (16, 256, 16)])
def test_tree_select_parity(torch, B, N, gamma):
    rng = np.random.default_rng(B * 7 + N)
    parent = np.empty((B, N), np.int32)
    for b in range(B):
        depth = []
        for s in range(N):
            cands = [-1] + [p for p in range(s) if depth[p] < gamma]
            parent[b, s] = rng.choice(cands)
            depth.append(1 if parent[b, s] < 0 else depth[parent[b, s]] + 1)
    conf = rng.random((B, N)).astype(np.float32)
    conf[:, ::5] = 0.5                                     # ties
    dev = "cuda"
    surv = torch.empty((B, N), dtype=torch.float32, device=dev)
    mask = torch.empty((B, N), dtype=torch.uint8, device=dev)
    exp = torch.empty(B, dtype=torch.float32, device=dev)
    st = torch.zeros(4, dtype=torch.int32, device=dev)
    for n in (0, 1, N // 2, N):
        _lib().spec_tree_select(torch.from_numpy(parent).to(dev), torch.from_numpy(conf).to(dev), n,
                                surv, mask, st, gamma, expected=exp)
        torch.cuda.synchronize()
        assert int(st[0]) == 0
        for b in range(B):
            assert np.array_equal(surv[b].cpu().numpy().view(np.uint32),
                                  TR.survival(parent[b], conf[b]).view(np.uint32))
            ref = TR.select(parent[b], conf[b], n)
            assert np.array_equal(mask[b].cpu().numpy().astype(bool), ref), (b, n)


def test_tree_select_rejects_bad_parents(torch):
    dev = "cuda"
    parent = torch.tensor([[-1, 0, 2]], dtype=torch.int32, device=dev)   # slot 2 is its own parent
    conf = torch.full((1, 3), 0.5, device=dev)
    surv = torch.empty((1, 3), device=dev)
    mask = torch.empty((1, 3), dtype=torch.uint8, device=dev)
    st = torch.zeros(4, dtype=torch.int32, device=dev)
    _lib().spec_tree_select(parent, conf, 2, surv, mask, st, 4)
    torch.cuda.synchronize()
    assert int(st[0]) & 128 and int(mask.sum()) == 0


@pytest.mark.parametrize("name,B,N,n", [("C0", None, 12, 8), ("C2", 6, 24, 12), ("C3", 2, 20, 10)])
def test_tree_cycle_parity(torch, name, B, N, n):
    from speculative_decoding_draft_04_gb300 import engine
    spec = W.config(name)
    w = W.make_workload(spec, 0, B=B)
    ti = W.make_tree_inputs(spec, w, N, 0)
    d = engine.DeviceWorkload.from_workload(w)
    t = engine.DeviceTree.from_inputs(ti, d, n)
    engine.tree_cycle(d, t)
    torch.cuda.synchronize()
    assert engine.status_words(t.status)[0] == 0
    mask = t.mask.cpu().numpy().astype(bool)
    tokens = t.tokens.cpu().numpy()
    q_tok = t.q_tok.cpu().numpy()
    acc, out, path = (x.cpu().numpy() for x in (t.accept_len, t.out_tokens, t.path))
    U, W1, W2 = W.to_f64(w.U, w.dtype), w.f64("W1"), w.f64("W2")
    for b in range(w.B):
        par = ti.parent[b]
        assert np.array_equal(mask[b], TR.select(par, ti.conf[b], n))
        dr = TR.draft_request(U[b], W1, W2, w.anchor[b], float(w.temperature[b]), par, mask[b],
                              ti.u_draft[b].astype(np.float64))
        near = dr.dist[mask[b]].min(initial=np.inf) < 1e-9
        if not near:
            assert np.array_equal(tokens[b], dr.tokens), b
            sel = mask[b]
            assert np.allclose(q_tok[b][sel], dr.q_tok[sel], atol=1e-5)
        # verification of the GPU's own draft
        tv = W.to_f64(ti.target[b], w.dtype)
        vr = TR.verify_request(tv, U[b], W1, W2, w.anchor[b], float(w.temperature[b]), par, mask[b],
                               tokens[b], ti.u_accept[b].astype(np.float64), float(ti.u_final[b]),
                               w.gamma)
        if vr.dmin >= 1e-9:
            assert acc[b] == len(vr.path), b
            assert np.array_equal(out[b], vr.out_tokens), b
            assert list(path[b][:acc[b]]) == vr.path and np.all(path[b][acc[b]:] == -1)
