"""Pins of the oracle's sparse-attention backward (NeMo _SparseAttention.backward:
grad_out -> dq, dk, dv) against things other than its own formulas: central
finite differences of the forward (on fp64 inputs, reduced to the loss
sum(out * grad_out)), and the closed form of a one-token document."""
import math

import numpy as np
import torch

import oracle

SCALE = 1.0 / math.sqrt(128)
H, G, D, BLOCK = 64, 4, 128, 128


def _bf16_round(x):
    return torch.from_numpy(x).to(torch.bfloat16).float().numpy().astype(np.float64)


def _q2k(cu, topk, rng):
    """Random valid q2k [G, T, topk]: ascending ids among each token's causal blocks, -1 padded."""
    T = cu[-1]
    q2k = np.full((G, T, topk), -1, dtype=np.int32)
    for d in range(len(cu) - 1):
        for t in range(cu[d], cu[d + 1]):
            nb = (t - cu[d]) // BLOCK + 1
            for g in range(G):
                ids = np.sort(rng.choice(nb, size=min(nb, topk), replace=False))
                q2k[g, t, :len(ids)] = ids
    return q2k


def _case(docs, topk, seed):
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(docs)]).astype(np.int32)
    T = int(cu[-1])
    q = _bf16_round(rng.standard_normal((T, H, D)))
    k = _bf16_round(rng.standard_normal((T, G, D)))
    v = _bf16_round(rng.standard_normal((T, G, D)))
    do = _bf16_round(rng.standard_normal((T, H, D)))
    return cu, q, k, v, do, _q2k(cu, topk, rng)


def _bf(x):
    return torch.from_numpy(x).to(torch.bfloat16)


def _grads(cu, q, k, v, do, q2k):
    return oracle.attend_prefill_backward(_bf(q), _bf(k), _bf(v), _bf(do), torch.from_numpy(cu),
                                          torch.from_numpy(q2k), SCALE)


def test_backward_matches_directional_finite_differences():
    # two documents, the longer spanning three blocks; top-2 of its blocks
    cu, q, k, v, do, q2k = _case([300, 70], topk=2, seed=0)
    dq, dk, dv = _grads(cu, q, k, v, do, q2k)
    rng = np.random.default_rng(1)
    loss = lambda q_, k_, v_: oracle.attend_loss_f64(q_, k_, v_, do, cu, q2k, SCALE)
    h = 1e-4
    for name, x, gx in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        d = rng.standard_normal(x.shape)
        args_p = {"q": q, "k": k, "v": v}
        args_m = {"q": q, "k": k, "v": v}
        args_p[name] = x + h * d
        args_m[name] = x - h * d
        fd = (loss(args_p["q"], args_p["k"], args_p["v"]) - loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
        an = float(np.sum(gx * d))
        assert abs(fd - an) <= 1e-6 * (1 + abs(an)), (name, fd, an)


def test_backward_matches_coordinate_finite_differences():
    cu, q, k, v, do, q2k = _case([200], topk=1, seed=2)
    dq, dk, dv = _grads(cu, q, k, v, do, q2k)
    loss = lambda q_, k_, v_: oracle.attend_loss_f64(q_, k_, v_, do, cu, q2k, SCALE)
    h = 1e-4
    picks = {"q": [(150, 17, 5), (3, 63, 127)], "k": [(0, 0, 0), (129, 3, 64)], "v": [(5, 2, 9), (199, 1, 100)]}
    for name, idx_list in picks.items():
        for idx in idx_list:
            args_p = {"q": q.copy(), "k": k.copy(), "v": v.copy()}
            args_m = {"q": q.copy(), "k": k.copy(), "v": v.copy()}
            args_p[name][idx] += h
            args_m[name][idx] -= h
            fd = (loss(args_p["q"], args_p["k"], args_p["v"]) - loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
            an = {"q": dq, "k": dk, "v": dv}[name][idx]
            assert abs(fd - an) <= 1e-6 * (1 + abs(an)), (name, idx, fd, an)


def test_backward_one_token_closed_form():
    # one key: softmax is 1, so out = v, dv = sum of the group's grad_out rows, dq = dk = 0
    cu, q, k, v, do, q2k = _case([1], topk=16, seed=3)
    dq, dk, dv = _grads(cu, q, k, v, do, q2k)
    assert np.all(dq == 0) and np.all(dk == 0)
    np.testing.assert_allclose(dv[0], do[0].reshape(G, H // G, D).sum(axis=1), rtol=0, atol=1e-12)
