"""qv_spec_sample (lossless rejection sampling at T > 0) against the oracle,
bit for bit: the accepted lengths and every emitted token, over seeds, for
draft distributions close to and far from the verifier's, at the full
Qwen3 vocabulary and at small ones."""
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


def _softmax32(x):
    x = x.astype(np.float64)
    e = np.exp(x - x.max(axis=1, keepdims=True))
    return (e / e.sum(axis=1, keepdims=True)).astype(np.float32)


def _case(B, gamma, V, mode, seed):
    rng = np.random.default_rng(seed)
    z = rng.normal(0.0, 2.0, (B * (gamma + 1), V)).astype(np.float32)
    rows = [b * (gamma + 1) + j for b in range(B) for j in range(gamma)]
    if mode == "close":
        zq = z[rows] + rng.normal(0.0, 0.3, (len(rows), V)).astype(np.float32)
    else:
        zq = rng.normal(0.0, 2.0, (len(rows), V)).astype(np.float32)
    q = _softmax32(zq) if rows else np.zeros((0, V), np.float32)
    qn = q.astype(np.float64)
    qn /= qn.sum(axis=1, keepdims=True) if rows else 1.0
    d = np.array([rng.choice(V, p=qn[i]) for i in range(len(rows))], dtype=np.int32).reshape(B, gamma)
    return z, d, q


def _run(qv, z, d, q, B, gamma, T, seed):
    V = z.shape[1]
    # the workspace needs no initialisation: hand it over full of junk
    g = torch.Generator(device="cuda").manual_seed(seed)
    ws = torch.randint(0, 256, (qv.qv_workspace_bytes(qv.QV_OP_SPEC_SAMPLE, B * (gamma + 1), 16, V),),
                       dtype=torch.uint8, device="cuda", generator=g)
    ln = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    out = torch.full((B, gamma + 1), -7, dtype=torch.int32, device="cuda")
    qv.qv_spec_sample(torch.from_numpy(z).cuda(), torch.from_numpy(d).cuda(), torch.from_numpy(q).cuda(),
                      T, seed, ln, out, ws)
    torch.cuda.synchronize()
    return np_(ln), np_(out)


CASES = [  # B, gamma, V, T, draft distribution
    (1, 4, 151936, 0.8, "close"),
    (3, 2, 1000, 1.0, "far"),
    (2, 0, 5000, 1.3, "close"),
    (4, 3, 64, 0.5, "close"),
    (8, 7, 3000, 1.0, "far"),
    (2, 3, 1, 1.0, "close"),
    (2, 2, 6145, 0.9, "far"),        # three full 2048-token chunks and a 1-token tail
    (1, 1, 2100000, 1.0, "close"),   # more chunks (1026) than draw-kernel threads
]


@pytest.mark.parametrize("B,gamma,V,T,mode", CASES)
def test_spec_sample(qv, oracle, B, gamma, V, T, mode):
    z, d, q = _case(B, gamma, V, mode, seed=B * 1000 + gamma * 10 + V % 97)
    lens = []
    for seed in range(8):
        ln, out = _run(qv, z, d, q, B, gamma, T, seed * 1000003 + 17)
        ln_ref, out_ref = oracle.spec_sample(z, d, q, B, gamma, T, seed * 1000003 + 17)
        assert np.array_equal(ln, ln_ref), (seed, ln, ln_ref)
        assert np.array_equal(out, out_ref), (seed, out, out_ref)
        lens.extend(ln.tolist())
    assert all(1 <= x <= gamma + 1 for x in lens)


def test_spec_sample_closed_cases(qv, oracle):
    """q equal to p keeps every draft; a draft with p(d) = 0 and a draft
    outside the vocabulary are never kept, and p(d) = 0 is never drawn."""
    B, gamma, V = 3, 4, 512
    z = np.zeros((B * (gamma + 1), V), np.float32)
    q = np.ones((B * gamma, V), np.float32)
    d = np.random.default_rng(1).integers(0, V, (B, gamma)).astype(np.int32)
    for seed in range(10):
        ln, _ = _run(qv, z, d, q, B, gamma, 1.0, seed)
        assert (ln == gamma + 1).all()
    rng = np.random.default_rng(2)
    z2 = rng.normal(0.0, 1.0, (B * (gamma + 1), V)).astype(np.float32)
    for b in range(B):
        z2[b * (gamma + 1), d[b, 0]] = -1000.0
    q2 = rng.uniform(0.01, 1.0, (B * gamma, V)).astype(np.float32)
    for seed in range(10):
        ln, out = _run(qv, z2, d, q2, B, gamma, 1.0, seed)
        ln_ref, out_ref = oracle.spec_sample(z2, d, q2, B, gamma, 1.0, seed)
        assert (ln == 1).all() and all(out[b, 0] != d[b, 0] for b in range(B))
        assert np.array_equal(ln, ln_ref) and np.array_equal(out, out_ref)
    d_bad = d.copy()
    d_bad[:, 0] = [V, -1, 1 << 30]
    ln, out = _run(qv, z, d_bad, q, B, gamma, 1.0, 5)
    assert (ln == 1).all() and ((out[:, 0] >= 0) & (out[:, 0] < V)).all()


def test_sampled_step_matches_oracle(qv, oracle):
    """A small stack's T > 0 step (layers, LM-head logits, qv_spec_sample in
    one graph) equals the oracle's sampling on the same logits."""
    from quantized_verification_gb300.stack import VerifyStack
    model = {"hidden": 256, "kv": 64, "ffn": 512, "layers": 2, "vocab": 3000}
    st = VerifyStack(model=model, B=2, gamma=3, seed=9)
    st.prepare_sampling(temperature=0.9, seed=77)
    g = st.capture_sampled()
    g.replay()
    torch.cuda.synchronize()
    ln_ref, out_ref = oracle.spec_sample(np_(st.logits), np_(st.q_drafts), np_(st.q), 2, 3, 0.9, 77)
    assert np.array_equal(np_(st.accept_len), ln_ref) and np.array_equal(np_(st.out_tokens), out_ref)
