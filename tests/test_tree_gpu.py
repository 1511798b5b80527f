"""qv_tree_accept (greedy verification of a draft tree) against the oracle,
bit for bit: accepted lengths, emitted tokens and the chosen node, on random
trees with tiny vocabularies (so that deep matching paths are common),
chain-shaped trees, invalid parents and the largest trees."""
import numpy as np
import pytest
import torch

from gpu_util import np_, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qv():
    require_gpu()
    from quantized_verification_gb300 import qv as _qv
    _qv.load()
    return _qv


def _run(qv, t, d, par):
    B, N = t.shape
    ln = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    out = torch.full((B, N), -7, dtype=torch.int32, device="cuda")
    node = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    qv.qv_tree_accept(torch.from_numpy(t).cuda(), torch.from_numpy(d).cuda(), torch.from_numpy(par).cuda(),
                      ln, out, best_node=node)
    torch.cuda.synchronize()
    return np_(ln), np_(out), np_(node)


@pytest.mark.parametrize("B,N,V", [(64, 1, 3), (64, 2, 2), (128, 16, 2), (32, 64, 3), (4, 1024, 2), (16, 37, 4)])
def test_tree_accept_random(qv, oracle, B, N, V):
    rng = np.random.default_rng(B * 31 + N)
    par = np.full((B, N), -1, np.int32)
    for i in range(1, N):
        par[:, i] = rng.integers(0, i, B)
    t = rng.integers(0, V, (B, N)).astype(np.int32)
    d = rng.integers(0, V, (B, N)).astype(np.int32)
    ln, out, node = _run(qv, t, d, par)
    ln_ref, out_ref, node_ref = oracle.tree_accept(t, d, par)
    assert np.array_equal(ln, ln_ref) and np.array_equal(out, out_ref) and np.array_equal(node, node_ref)
    if N >= 16:
        assert ln.max() >= 3            # deep matching paths are exercised


def test_tree_accept_chain_and_invalid_parents(qv, oracle):
    """A chain tree gives qv_accept's result; parents outside [0, i) make a
    node (and its subtree) unacceptable, on both sides alike."""
    B, N, V = 32, 8, 2
    rng = np.random.default_rng(5)
    t = rng.integers(0, V, (B, N)).astype(np.int32)
    d = rng.integers(0, V, (B, N)).astype(np.int32)
    par = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
    ln, out, _ = _run(qv, t, d, par)
    ln_ref, out_ref = oracle.accept(t, d[:, 1:], B, N - 1)
    assert np.array_equal(ln, ln_ref) and np.array_equal(out, out_ref)
    bad = par.copy()
    bad[:, 3] = 5            # a parent after the node
    bad[:, 6] = -4           # a negative parent
    ln, out, node = _run(qv, t, d, bad)
    ln_ref, out_ref, node_ref = oracle.tree_accept(t, d, bad)
    assert np.array_equal(ln, ln_ref) and np.array_equal(out, out_ref) and np.array_equal(node, node_ref)
    assert (node != 3).all() and (node != 6).all()
