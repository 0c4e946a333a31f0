"""Pins of the fp64 oracle against things fixed outside of it.

No page prints a worked numeric example of the layer, so every pin here is a
closed form, an invariant, a library routine the oracle does not use, or brute
force (finite differences). Each one is chosen so that a plausible slip in the
oracle (a dropped term, a sign, a transposed operand, a mean instead of a sum,
apply/update in the wrong order, a wrong norm axis) fails at least one test.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import ttt_oracle as orc

RNG = np.random.default_rng(1234)


def _rand_weights(fast_net, d, dh, rng, scale=1.0):
    if fast_net == "swiglu":
        return (rng.standard_normal((dh, d)) * scale / np.sqrt(d),
                rng.standard_normal((d, dh)) * scale / np.sqrt(dh),
                rng.standard_normal((dh, d)) * scale / np.sqrt(d))
    return (rng.standard_normal((d, d)) / np.sqrt(d),)


def _loss_from_definition(fast_net, loss, W, K, V, eta):
    """sum_t eta_t l_t with l_t = -f(k_t).v_t or 1/2 ||f(k_t) - v_t||^2."""
    f = orc.swiglu_apply(W, K) if fast_net == "swiglu" else orc.linear_apply(W, K)
    if loss == "ip":
        per = -(f * V).sum(axis=1)
    else:
        per = 0.5 * ((f - V) ** 2).sum(axis=1)
    return float((eta * per).sum())


@pytest.mark.parametrize("fast_net", ["swiglu", "linear"])
@pytest.mark.parametrize("loss", ["ip", "mse"])
def test_gradient_matches_central_differences(fast_net, loss):
    """Brute force: every gradient entry against a central difference (h = 1e-6)."""
    rng = np.random.default_rng(7)
    d, dh, C = 4, 8, 3
    W = _rand_weights(fast_net, d, dh, rng, scale=1.5)
    K = rng.standard_normal((C, d))
    V = rng.standard_normal((C, d))
    eta = rng.uniform(0.1, 1.0, C)
    fn = orc.swiglu_grad if fast_net == "swiglu" else orc.linear_grad
    G = fn(W, K, V, eta, loss)
    h = 1e-6
    for j, Wj in enumerate(W):
        fd = np.zeros_like(Wj)
        for idx in np.ndindex(*Wj.shape):
            Wp = [w.copy() for w in W]
            Wm = [w.copy() for w in W]
            Wp[j][idx] += h
            Wm[j][idx] -= h
            fd[idx] = (_loss_from_definition(fast_net, loss, Wp, K, V, eta)
                       - _loss_from_definition(fast_net, loss, Wm, K, V, eta)) / (2 * h)
        err = np.abs(fd - G[j]).max() / np.abs(G[j]).max()
        assert err < 1e-7, (j, err)


@pytest.mark.parametrize("loss", ["ip", "mse"])
def test_swiglu_gradient_matches_torch_autograd(loss):
    """torch (a different library, with its own silu) differentiates the same loss."""
    rng = np.random.default_rng(11)
    d, dh, C = 6, 10, 9
    W = _rand_weights("swiglu", d, dh, rng, scale=2.0)
    K = rng.standard_normal((C, d))
    V = rng.standard_normal((C, d))
    eta = rng.uniform(0.0, 0.3, C)
    tw = [torch.tensor(w, dtype=torch.float64, requires_grad=True) for w in W]
    tk, tv, te = (torch.tensor(x, dtype=torch.float64) for x in (K, V, eta))
    f = F.linear(F.silu(F.linear(tk, tw[0])) * F.linear(tk, tw[2]), tw[1])
    per = -(f * tv).sum(1) if loss == "ip" else 0.5 * ((f - tv) ** 2).sum(1)
    (te * per).sum().backward()
    G = orc.swiglu_grad(W, K, V, eta, loss)
    for j in range(3):
        ref = tw[j].grad.numpy()
        assert np.abs(G[j] - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


def test_swiglu_forward_matches_torch():
    rng = np.random.default_rng(3)
    d, dh = 16, 40
    W = _rand_weights("swiglu", d, dh, rng, scale=3.0)
    X = rng.standard_normal((25, d))
    tw = [torch.tensor(w, dtype=torch.float64) for w in W]
    tx = torch.tensor(X, dtype=torch.float64)
    ref = F.linear(F.silu(F.linear(tx, tw[0])) * F.linear(tx, tw[2]), tw[1]).numpy()
    assert np.abs(orc.swiglu_apply(W, X) - ref).max() <= 1e-13 * np.abs(ref).max()


@pytest.mark.parametrize("fast_net", ["swiglu", "linear"])
def test_chunk_gradient_is_sum_of_token_gradients(fast_net):
    """LaCT page §2.1: the update uses the gradient SUMMED over the chunk's tokens."""
    rng = np.random.default_rng(5)
    d, dh, C = 8, 16, 37
    W = _rand_weights(fast_net, d, dh, rng)
    K = rng.standard_normal((C, d))
    V = rng.standard_normal((C, d))
    eta = rng.uniform(0, 0.1, C)
    cfg = orc.OracleCfg(chunk=C, fast_net=fast_net, loss="mse")
    G = orc.chunk_grad(cfg, W, K, V, eta)
    Gb = orc.chunk_grad(cfg, W, K, V, eta, block=5)
    per = [orc.chunk_grad(cfg, W, K[t:t + 1], V[t:t + 1], eta[t:t + 1]) for t in range(C)]
    for j in range(len(W)):
        s = sum(p[j] for p in per)
        assert np.abs(G[j] - s).max() <= 1e-12 * np.abs(s).max()
        assert np.abs(Gb[j] - s).max() <= 1e-12 * np.abs(s).max()


def test_linear_mse_chunk1_is_delta_rule():
    """Chunk of one token, linear net, MSE, plain SGD: the delta rule
    W <- W - eta (W k - v) k^T, with o_t read from W before token t's update."""
    rng = np.random.default_rng(9)
    d, T = 5, 23
    W0 = rng.standard_normal((d, d)) / np.sqrt(d)
    Q, K, V = (rng.standard_normal((T, d)) for _ in range(3))
    eta = rng.uniform(0, 0.2, T)
    cfg = orc.OracleCfg(chunk=1, fast_net="linear", loss="mse", muon=False, wnorm=False)
    O, (Wf,) = orc.ttt_head(cfg, Q, K, V, eta, (W0,))
    W = W0.copy()
    Oref = np.zeros((T, d))
    for t in range(T):
        Oref[t] = W @ Q[t]
        W = W - eta[t] * np.outer(W @ K[t] - V[t], K[t])
    assert np.abs(O - Oref).max() <= 1e-12
    assert np.abs(Wf - W).max() <= 1e-12


def test_linear_mse_chunk_of_orthonormal_keys_memorises_it():
    """Linear net, MSE, SGD, unit rates, each chunk's keys orthonormal (C <= d):
    the chunk-summed step is then an exact least-squares solve on the keys' span,
    so the updated W sends every key of the chunk to its value and leaves the
    orthogonal complement untouched. In shifted order the next chunk's queries
    read that W: queries equal to the previous chunk's keys return its values."""
    rng = np.random.default_rng(33)
    d, C, n = 8, 4, 3
    T = C * n
    W0 = rng.standard_normal((d, d)) / np.sqrt(d)
    K = np.concatenate([np.linalg.qr(rng.standard_normal((d, C)))[0].T for _ in range(n)])
    V = rng.standard_normal((T, d))
    Q = rng.standard_normal((T, d))
    Q[C:] = K[:-C]                     # chunk c+1 asks for chunk c's keys
    cfg = orc.OracleCfg(chunk=C, fast_net="linear", loss="mse", muon=False, wnorm=False)
    O, (Wf,) = orc.ttt_head(cfg, Q, K, V, np.ones(T), (W0,))
    assert np.abs(O[:C] - Q[:C] @ W0.T).max() <= 1e-12
    assert np.abs(O[C:] - V[:-C]).max() <= 1e-12
    Kl = K[-C:]
    assert np.abs(Kl @ Wf.T - V[-C:]).max() <= 1e-12
    # the last step moved W only on the span of the last chunk's keys
    _, (Wp,) = orc.ttt_head(cfg, Q[:-C], K[:-C], V[:-C], np.ones(T - C), (W0,))
    u = rng.standard_normal(d)
    u -= Kl.T @ (Kl @ u)
    assert np.abs(Wf @ u - Wp @ u).max() <= 1e-12


@pytest.mark.parametrize("mask", [None, [1, 0, 1, 1, 0], [0, 1, 0, 1, 0]])
def test_linear_ip_is_block_shifted_linear_attention(mask):
    """Linear net, inner-product loss, SGD: o_t = W0 q_t + sum over tokens s of
    UPDATED chunks strictly before t's chunk of eta_s v_s (k_s . q_t)."""
    rng = np.random.default_rng(21)
    d, C, T = 6, 4, 19     # ragged last chunk
    W0 = rng.standard_normal((d, d))
    Q, K, V = (rng.standard_normal((T, d)) for _ in range(3))
    eta = rng.uniform(0, 0.5, T)
    cfg = orc.OracleCfg(chunk=C, fast_net="linear", loss="ip", muon=False, wnorm=False,
                        mask=mask)
    O, (Wf,) = orc.ttt_head(cfg, Q, K, V, eta, (W0,))
    m = mask or [1] * 5
    upd = np.array([m[s // C] for s in range(T)], dtype=float)
    Oref = np.zeros((T, d))
    for t in range(T):
        start = (t // C) * C
        acc = W0 @ Q[t]
        for s in range(start):
            acc = acc + upd[s] * eta[s] * V[s] * (K[s] @ Q[t])
        Oref[t] = acc
    assert np.abs(O - Oref).max() <= 1e-12
    Wref = W0 + sum(upd[s] * eta[s] * np.outer(V[s], K[s]) for s in range(T))
    assert np.abs(Wf - Wref).max() <= 1e-12


def test_linear_ip_single_chunk_is_noncausal_linear_attention():
    """Single-chunk update-then-apply (LaCT page §3.1): every query sees every key."""
    rng = np.random.default_rng(22)
    d, T = 7, 30
    W0 = rng.standard_normal((d, d))
    Q, K, V = (rng.standard_normal((T, d)) for _ in range(3))
    eta = rng.uniform(0, 0.5, T)
    cfg = orc.OracleCfg(chunk=T, fast_net="linear", loss="ip", mode="single",
                        muon=False, wnorm=False)
    O, _ = orc.ttt_head(cfg, Q, K, V, eta, (W0,))
    Oref = Q @ W0.T + ((Q @ K.T) * eta[None, :]) @ V
    assert np.abs(O - Oref).max() <= 1e-12


NS = (3.4445, -4.7750, 2.0315)


def _phi5(x):
    a, b, c = NS
    for _ in range(5):
        x = a * x + b * x ** 3 + c * x ** 5
    return x


@pytest.mark.parametrize("shape", [(8, 20), (20, 8), (12, 12), (64, 128)])
def test_newton_schulz_closed_form_through_svd(shape):
    """The iteration acts on singular values only: G = U S V^T gives
    NS5(G) = U phi^5(S / (||G||_F + eps)) V^T, phi(x) = a x + b x^3 + c x^5."""
    rng = np.random.default_rng(shape[0] * 100 + shape[1])
    G = rng.standard_normal(shape) * 0.01
    U, S, Vt = np.linalg.svd(G, full_matrices=False)
    ref = (U * _phi5(S / (np.linalg.norm(S) + 1e-7))) @ Vt
    out = orc.newton_schulz(G, 5, *NS, 1e-7)
    assert np.abs(out - ref).max() <= 1e-10 * np.abs(ref).max()


def test_newton_schulz_singular_values_near_one():
    """LaCT page §2.2.1: Muon turns the gradient into an (approximately)
    orthogonal matrix. phi^5 maps [3e-3, 1] into [0.6, 1.25]; real chunk
    gradients of the workload shapes land there."""
    xs = np.linspace(3e-3, 1.0, 20001)
    y = _phi5(xs)
    assert y.min() > 0.6 and y.max() < 1.25
    rng = np.random.default_rng(2)
    d, dh, C = 32, 64, 256
    W = _rand_weights("swiglu", d, dh, rng)
    K = rng.standard_normal((C, d))
    K /= np.linalg.norm(K, axis=1, keepdims=True)
    V = rng.standard_normal((C, d))
    eta = 0.01 / (1 + np.exp(-rng.standard_normal(C)))
    for Gj in orc.swiglu_grad(W, K, V, eta, "ip"):
        s_in = np.linalg.svd(Gj, compute_uv=False)
        s_in = s_in / (np.linalg.norm(s_in) + 1e-7)
        s_out = np.linalg.svd(orc.newton_schulz(Gj, 5, *NS, 1e-7), compute_uv=False)
        keep = s_in >= 3e-3
        assert keep.sum() >= min(Gj.shape) // 2
        assert s_out[keep].min() > 0.6 and s_out[keep].max() < 1.25


@pytest.mark.parametrize("shape", [(6, 5), (5, 5), (4, 7)])
def test_weight_norm_restores_row_norms_and_keeps_directions(shape):
    rng = np.random.default_rng(4)
    W = (rng.standard_normal(shape),)
    G = (rng.standard_normal(shape),)
    n0 = [np.abs(rng.standard_normal(shape[0])) + 0.1]
    cfg = orc.OracleCfg(chunk=1, fast_net="linear", muon=False, wnorm=True, step=0.7)
    (Wn,) = orc.update(cfg, W, G, n0)
    raw = W[0] - 0.7 * G[0]
    assert np.abs(np.linalg.norm(Wn, axis=1) - n0[0]).max() <= 1e-13
    ratio = Wn / raw
    assert (ratio > 0).all()
    assert np.abs(ratio - ratio[:, :1]).max() <= 1e-12   # one positive scale per row


def _orthogonal(n, rng):
    q, r = np.linalg.qr(rng.standard_normal((n, n)))
    return q * np.sign(np.diag(r))


@pytest.mark.parametrize("loss,momentum,mode,per_matrix", [
    ("ip", 0.0, "shifted", False), ("mse", 0.0, "shifted", False), ("ip", 0.5, "shifted", False),
    ("mse", 0.5, "shifted", True), ("ip", 0.0, "single", True), ("mse", 0.0, "single", False)])
def test_muon_layer_is_equivariant_under_rotations_and_hidden_permutations(loss, momentum, mode, per_matrix):
    """The whole SwiGLU + Muon + weight-norm chain: shifted chunks under a mask, or one
    chunk in single mode; one rate per token, or one per token and matrix.
    Rotate the input space (R, any orthogonal), sign-permute the output space (S) and
    permute the hidden units (P): q, k -> R q, R k;  v -> S v;  W1, W3 -> P W (R^T);
    W2 -> S W2 P^T. Then f'(R x) = S f(x), both losses are unchanged, every gradient
    moves the same way as its matrix, Newton-Schulz commutes with orthogonal factors on
    either side, and the rows of every matrix keep their norms (up to the order), so
    O' = O S^T and each final matrix is the transformed final matrix. A weight norm over
    the wrong axis, or a Newton-Schulz scaling by anything but an orthogonally invariant
    norm, breaks it."""
    rng = np.random.default_rng(77)
    d, dh, C, T = 6, 10, 5, 17
    W = _rand_weights("swiglu", d, dh, rng, scale=2.0)
    Q, K, V = (rng.standard_normal((T, d)) for _ in range(3))
    eta = rng.uniform(0.0, 0.3, (T, 3) if per_matrix else T)
    R = _orthogonal(d, rng)
    S = np.eye(d)[rng.permutation(d)] * rng.choice([-1.0, 1.0], d)[:, None]
    P = np.eye(dh)[rng.permutation(dh)]
    cfg = orc.OracleCfg(chunk=C if mode == "shifted" else T, loss=loss, mode=mode, muon=True, wnorm=True,
                        step=0.7, mask=[1, 0, 1, 1] if mode == "shifted" else None, momentum=momentum)
    O, (W1, W2, W3) = orc.ttt_head(cfg, Q, K, V, eta, W)
    Wt = (P @ W[0] @ R.T, S @ W[1] @ P.T, P @ W[2] @ R.T)
    Ot, (W1t, W2t, W3t) = orc.ttt_head(cfg, Q @ R.T, K @ R.T, V @ S.T, eta, Wt)
    assert np.abs(Ot - O @ S.T).max() <= 1e-10 * np.abs(O).max()
    assert np.abs(W1t - P @ W1 @ R.T).max() <= 1e-10
    assert np.abs(W2t - S @ W2 @ P.T).max() <= 1e-10
    assert np.abs(W3t - P @ W3 @ R.T).max() <= 1e-10


def _quintic_at_one(iters, a, b, c, x=1.0):
    for _ in range(iters):
        x = a * x + b * x ** 3 + c * x ** 5
    return x


@pytest.mark.parametrize("wnorm", [False, True])
def test_muon_step_on_one_token_moves_along_the_unit_gradient(wnorm):
    """A one-token chunk gives a rank-one gradient G = sigma u v^T for each matrix, and
    Newton-Schulz of a rank-one matrix is its unit direction times the scalar quintic
    iterated from 1: W <- W - step * phi^5(1) * G / ||G||_F (then the row norm). The
    rate scales G but not the step (Muon discards the gradient's size). G here is torch
    autograd of eta * l(f(k), v) on the oracle-independent torch forward."""
    rng = np.random.default_rng(78)
    d, dh = 7, 12
    W = _rand_weights("swiglu", d, dh, rng, scale=2.0)
    Q, K, V = (rng.standard_normal((2, d)) for _ in range(3))
    eta = np.array([0.37, 0.2])
    step = 0.05
    cfg = orc.OracleCfg(chunk=1, loss="ip", muon=True, wnorm=wnorm, step=step, ns_eps=0.0)
    O, Wf = orc.ttt_head(cfg, Q, K, V, eta, W)

    tw = [torch.tensor(w, dtype=torch.float64, requires_grad=True) for w in W]
    k, v = (torch.tensor(x[0], dtype=torch.float64) for x in (K, V))
    f = F.linear(F.silu(F.linear(k, tw[0])) * F.linear(k, tw[2]), tw[1])
    (-eta[0] * (f * v).sum()).backward()
    s = _quintic_at_one(cfg.ns_iters, *cfg.ns_coef)
    W1 = []
    for w, t in zip(W, tw):
        g = t.grad.numpy()
        assert np.linalg.matrix_rank(g) == 1
        nw = w - step * s * g / np.linalg.norm(g)
        if wnorm:
            nw = nw * (np.linalg.norm(w, axis=1) / np.linalg.norm(nw, axis=1))[:, None]
        W1.append(nw)
    _, Wk = orc.ttt_head(cfg, Q[:1], K[:1], V[:1], eta[:1], W)
    for a, b in zip(Wk, W1):
        assert np.abs(a - b).max() <= 1e-12
    # the second token reads the once-updated weights (shifted order)
    t1 = [torch.tensor(w, dtype=torch.float64) for w in W1]
    q = torch.tensor(Q[1], dtype=torch.float64)
    o1 = F.linear(F.silu(F.linear(q, t1[0])) * F.linear(q, t1[2]), t1[1]).numpy()
    assert np.abs(O[1] - o1).max() <= 1e-12 * np.abs(o1).max()


@pytest.mark.parametrize("muon", [False, True])
def test_layer_keeps_every_row_norm_of_w0(muon):
    rng = np.random.default_rng(6)
    d, dh, C, T = 8, 16, 5, 23
    W0 = _rand_weights("swiglu", d, dh, rng)
    Q, K, V = (rng.standard_normal((T, d)) for _ in range(3))
    eta = rng.uniform(0, 0.1, T)
    cfg = orc.OracleCfg(chunk=C, muon=muon, wnorm=True)
    _, Wf = orc.ttt_head(cfg, Q, K, V, eta, W0)
    for w0, wf in zip(W0, Wf):
        assert np.abs(np.linalg.norm(wf, axis=1) - np.linalg.norm(w0, axis=1)).max() <= 1e-12
        assert np.abs(wf - w0).max() > 1e-3            # it did move


def test_one_sgd_chunk_steps_against_the_brute_force_gradient():
    """Update direction and step: W1 = W0 - step * grad, grad by finite differences."""
    rng = np.random.default_rng(8)
    d, dh, C = 3, 5, 4
    W0 = _rand_weights("swiglu", d, dh, rng)
    Q, K, V = (rng.standard_normal((C, d)) for _ in range(3))
    eta = rng.uniform(0.1, 0.5, C)
    cfg = orc.OracleCfg(chunk=C, muon=False, wnorm=False, step=0.5)
    _, Wf = orc.ttt_head(cfg, Q, K, V, eta, W0)
    h = 1e-6
    for j in range(3):
        fd = np.zeros_like(W0[j])
        for idx in np.ndindex(*W0[j].shape):
            Wp = [w.copy() for w in W0]
            Wm = [w.copy() for w in W0]
            Wp[j][idx] += h
            Wm[j][idx] -= h
            fd[idx] = (_loss_from_definition("swiglu", "ip", Wp, K, V, eta)
                       - _loss_from_definition("swiglu", "ip", Wm, K, V, eta)) / (2 * h)
        assert np.abs(Wf[j] - (W0[j] - 0.5 * fd)).max() <= 1e-8


@pytest.mark.parametrize("muon", [False, True])
def test_shifted_chunks_do_not_leak_the_future(muon):
    """LaCT page §3.2 (shifted block-causal mask): outputs of chunks before j do
    not change when anything of chunk j changes, and chunk j's own outputs do
    not see its own keys and values."""
    rng = np.random.default_rng(10)
    d, dh, C, T = 8, 16, 6, 30
    W0 = _rand_weights("swiglu", d, dh, rng)
    Q, K, V = (rng.standard_normal((T, d)) for _ in range(3))
    eta = rng.uniform(0, 0.1, T)
    cfg = orc.OracleCfg(chunk=C, muon=muon, wnorm=True)
    O, _ = orc.ttt_head(cfg, Q, K, V, eta, W0)
    j = 3
    sl = slice(j * C, (j + 1) * C)
    Q2, K2, V2 = Q.copy(), K.copy(), V.copy()
    K2[sl] += 1.0
    V2[sl] -= 2.0
    O2, _ = orc.ttt_head(cfg, Q2, K2, V2, eta, W0)
    assert np.array_equal(O2[:(j + 1) * C], O[:(j + 1) * C])
    assert np.abs(O2[(j + 1) * C:] - O[(j + 1) * C:]).max() > 1e-6
    Q2[sl] += 1.0
    O3, _ = orc.ttt_head(cfg, Q2, K2, V2, eta, W0)
    assert np.array_equal(O3[:j * C], O[:j * C])


def test_no_update_is_the_plain_swiglu_mlp():
    rng = np.random.default_rng(12)
    d, dh, C, T = 8, 16, 4, 16
    W0 = _rand_weights("swiglu", d, dh, rng)
    Q, K, V = (rng.standard_normal((T, d)) for _ in range(3))
    eta = rng.uniform(0, 0.1, T)
    cfg = orc.OracleCfg(chunk=C, mask=[0, 0, 0, 0])
    O, Wf = orc.ttt_head(cfg, Q, K, V, eta, W0)
    tw = [torch.tensor(w) for w in W0]
    ref = F.linear(F.silu(F.linear(torch.tensor(Q), tw[0])) * F.linear(torch.tensor(Q), tw[2]),
                   tw[1]).numpy()
    assert np.abs(O - ref).max() <= 1e-13 * np.abs(ref).max()
    assert all(np.array_equal(a, b) for a, b in zip(Wf, W0))


def test_video_mask_skips_noisy_chunks():
    """LaCT page §3.3: fast weights change only after the clean-frame chunks."""
    rng = np.random.default_rng(13)
    d, dh, C, T = 8, 16, 4, 16
    W0 = _rand_weights("swiglu", d, dh, rng)
    Q, K, V = (rng.standard_normal((T, d)) for _ in range(3))
    eta = rng.uniform(0, 0.1, T)
    cfg = orc.OracleCfg(chunk=C, mask=[0, 1, 0, 1])
    O, _ = orc.ttt_head(cfg, Q, K, V, eta, W0)
    assert np.abs(O[C:2 * C] - orc.swiglu_apply(W0, Q[C:2 * C])).max() == 0.0
    # chunk 2 sees exactly one update, the one of chunk 1
    W1 = orc.update(cfg, W0, orc.chunk_grad(cfg, W0, K[C:2 * C], V[C:2 * C], eta[C:2 * C]),
                    [np.linalg.norm(w, axis=1) for w in W0])
    assert np.abs(O[2 * C:3 * C] - orc.swiglu_apply(W1, Q[2 * C:3 * C])).max() <= 1e-13


def test_single_chunk_is_permutation_invariant():
    rng = np.random.default_rng(14)
    d, dh, T = 8, 16, 40
    W0 = _rand_weights("swiglu", d, dh, rng)
    Q, K, V = (rng.standard_normal((T, d)) for _ in range(3))
    eta = rng.uniform(0, 0.1, T)
    cfg = orc.OracleCfg(chunk=T, mode="single")
    O, Wf = orc.ttt_head(cfg, Q, K, V, eta, W0)
    p = rng.permutation(T)
    O2, Wf2 = orc.ttt_head(cfg, Q[p], K[p], V[p], eta[p], W0)
    for a, b in zip(Wf, Wf2):
        assert np.abs(a - b).max() <= 1e-12
    assert np.abs(O2 - O[p]).max() <= 1e-12


@pytest.mark.parametrize("wnorm", [False, True])
def test_resume_at_a_chunk_boundary(wnorm):
    """Two calls split at a chunk boundary, the second starting from the first's
    final weights, equal one call (W_final is the layer's whole state)."""
    rng = np.random.default_rng(15)
    d, dh, C, T = 8, 16, 5, 30
    W0 = _rand_weights("swiglu", d, dh, rng)
    Q, K, V = (rng.standard_normal((T, d)) for _ in range(3))
    eta = rng.uniform(0, 0.1, T)
    cfg = orc.OracleCfg(chunk=C, wnorm=wnorm)
    O, Wf = orc.ttt_head(cfg, Q, K, V, eta, W0)
    s = 3 * C
    Oa, Wa = orc.ttt_head(cfg, Q[:s], K[:s], V[:s], eta[:s], W0)
    Ob, Wb = orc.ttt_head(cfg, Q[s:], K[s:], V[s:], eta[s:], Wa)
    tol = 1e-12 if wnorm else 0.0
    assert np.abs(np.concatenate([Oa, Ob]) - O).max() <= tol
    for a, b in zip(Wb, Wf):
        assert np.abs(a - b).max() <= tol


def test_toy_scalar_ttt_on_a_noisy_sinusoid():
    """Tutorial page §10 project: scalar w, MSE on predicting x_t from x_{t-1},
    SGD with lr 0.01, update then predict. With d = 1 the layer is the scalar
    recurrence w <- w - 0.01 (w x_{t-1} - x_t) x_{t-1}."""
    rng = np.random.default_rng(16)
    t = np.arange(1001)
    x = np.sin(0.05 * t) + 0.05 * rng.standard_normal(t.size)
    K = x[:-1, None]
    V = x[1:, None]
    eta = np.full(1000, 0.01)
    cfg = orc.OracleCfg(chunk=1, fast_net="linear", loss="mse", muon=False, wnorm=False)
    O, (Wf,) = orc.ttt_head(cfg, K, K, V, eta, (np.zeros((1, 1)),))
    w = 0.0
    pred = []
    for i in range(1000):
        pred.append(w * K[i, 0])
        w -= 0.01 * (w * K[i, 0] - V[i, 0]) * K[i, 0]
    assert np.isfinite(O).all()
    assert np.abs(O[:, 0] - np.array(pred)).max() <= 1e-12
    assert abs(Wf[0, 0] - w) <= 1e-12
    # the adapted scalar predicts better than the initial w = 0 on the last half
    assert ((O[500:, 0] - V[500:, 0]) ** 2).mean() < (V[500:, 0] ** 2).mean()


# ------------------------------------------------------------------ momentum, per-matrix rates
@pytest.mark.parametrize("mu", [0.5, 0.9])
def test_linear_ip_momentum_is_a_geometric_sum_of_chunk_gradients(mu):
    """Linear net, inner-product loss, momentum optimiser (Muon off, no weight
    norm): a chunk's gradient g_c = -sum_s eta_s v_s k_s^T does not depend on W,
    the buffer after the i-th update is sum_{k<=i} mu^(i-k) g_(k), so after m
    updates W = W0 - step * sum_k g_(k) (1 - mu^(m-k+1)) / (1 - mu): a geometric
    series written out, not the recursion. Skipped chunks leave the buffer as is."""
    rng = np.random.default_rng(31)
    d, C, T, step = 5, 4, 23, 0.7
    mask = [1, 0, 1, 1, 0, 1]
    W0 = rng.standard_normal((d, d))
    Q, K, V = (rng.standard_normal((T, d)) for _ in range(3))
    eta = rng.uniform(0, 0.5, T)
    cfg = orc.OracleCfg(chunk=C, fast_net="linear", loss="ip", muon=False, wnorm=False,
                        mask=mask, momentum=mu, step=step)
    O, (Wf,) = orc.ttt_head(cfg, Q, K, V, eta, (W0,))
    n = (T + C - 1) // C
    g = [-sum(eta[s] * np.outer(V[s], K[s]) for s in range(c * C, min(T, (c + 1) * C))) for c in range(n)]
    upd = [c for c in range(n) if mask[c]]

    def weights_after(m):  # after the first m updates
        return W0 - step * sum(g[upd[k]] * (1 - mu ** (m - k)) / (1 - mu) for k in range(m))

    for t in range(T):
        m = sum(1 for c in upd if c < t // C)
        assert np.abs(O[t] - weights_after(m) @ Q[t]).max() <= 1e-12
    assert np.abs(Wf - weights_after(len(upd))).max() <= 1e-12


def test_momentum_feeds_newton_schulz():
    """With Muon on, the buffer (not the gradient) is orthogonalised: when the
    second chunk's rates are all zero its gradient vanishes, the buffer is
    mu * (first gradient), and Newton-Schulz of it is that of the first gradient
    (its normalisation removes the scale, up to eps). Momentum applied after
    Newton-Schulz would step by mu times that instead."""
    rng = np.random.default_rng(32)
    d, dh, C = 4, 8, 6
    T = 2 * C
    W0 = _rand_weights("swiglu", d, dh, rng)
    Q, K, V = (rng.standard_normal((T, d)) for _ in range(3))
    eta = np.concatenate([rng.uniform(0.1, 0.5, C), np.zeros(C)])
    cfg = orc.OracleCfg(chunk=C, mode="shifted", muon=True, wnorm=False, momentum=0.6)
    _, W = orc.ttt_head(cfg, Q, K, V, eta, W0)
    G = orc.chunk_grad(cfg, W0, K[:C], V[:C], eta[:C])
    for j in range(3):
        U = orc.newton_schulz(G[j], 5, *cfg.ns_coef, 1e-7)
        assert np.abs(W[j] - (W0[j] - 2.0 * U)).max() <= 1e-6 * np.abs(U).max()


def test_per_matrix_rates_weight_each_matrix_by_its_own_column():
    """eta [n, 3]: matrix j's gradient is sum_t eta_(t,j) times token t's own
    gradient (the gradient with a one-hot weight on t), by brute force."""
    rng = np.random.default_rng(33)
    d, dh, C = 4, 8, 5
    W = _rand_weights("swiglu", d, dh, rng)
    K, V = rng.standard_normal((C, d)), rng.standard_normal((C, d))
    eta3 = rng.uniform(0.0, 1.0, (C, 3))
    cfg = orc.OracleCfg(chunk=C)
    G = orc.chunk_grad(cfg, W, K, V, eta3)
    for j in range(3):
        ref = sum(eta3[t, j] * orc.swiglu_grad(W, K[t:t + 1], V[t:t + 1], np.ones(1), "ip")[j]
                  for t in range(C))
        assert np.abs(G[j] - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


def test_per_matrix_rates_equal_to_the_shared_rate_give_the_same_layer():
    rng = np.random.default_rng(34)
    d, dh, C, T = 4, 8, 5, 17
    W0 = _rand_weights("swiglu", d, dh, rng)
    Q, K, V = (rng.standard_normal((T, d)) for _ in range(3))
    eta = rng.uniform(0.0, 0.3, T)
    cfg = orc.OracleCfg(chunk=C, muon=True, wnorm=True)
    O1, W1 = orc.ttt_head(cfg, Q, K, V, eta, W0)
    O3, W3 = orc.ttt_head(cfg, Q, K, V, np.stack([eta] * 3, axis=1), W0)
    assert np.array_equal(O1, O3) and all(np.array_equal(a, b) for a, b in zip(W1, W3))


def test_a_zero_rate_leaves_its_matrix_unchanged():
    """SGD without weight norm: a matrix whose rates are all zero never moves,
    the others do."""
    rng = np.random.default_rng(35)
    d, dh, C, T = 4, 8, 5, 15
    W0 = _rand_weights("swiglu", d, dh, rng)
    Q, K, V = (rng.standard_normal((T, d)) for _ in range(3))
    eta3 = rng.uniform(0.1, 0.3, (T, 3))
    eta3[:, 1] = 0.0
    cfg = orc.OracleCfg(chunk=C, muon=False, wnorm=False)
    _, W = orc.ttt_head(cfg, Q, K, V, eta3, W0)
    assert np.array_equal(W[1], W0[1])
    assert np.abs(W[0] - W0[0]).max() > 1e-3 and np.abs(W[2] - W0[2]).max() > 1e-3


# ---------------------------------------------------------------- inclusive (per-token) order
def test_inclusive_chunk1_linear_mse_is_the_delta_rule_read_after_the_update():
    """Tutorial page §3: theta_t = theta_{t-1} - eta grad l(theta_{t-1}; x_t), then
    h_t = f(x_t; theta_t). Chunks of one token, linear net, MSE: the delta rule
    with o_t read AFTER token t's own update."""
    rng = np.random.default_rng(31)
    d, T = 5, 21
    W0 = rng.standard_normal((d, d)) / np.sqrt(d)
    Q, K, V = (rng.standard_normal((T, d)) for _ in range(3))
    eta = rng.uniform(0, 0.2, T)
    cfg = orc.OracleCfg(chunk=1, fast_net="linear", loss="mse", mode="inclusive", muon=False, wnorm=False)
    O, (Wf,) = orc.ttt_head(cfg, Q, K, V, eta, (W0,))
    W = W0.copy()
    Oref = np.zeros((T, d))
    for t in range(T):
        W = W - eta[t] * np.outer(W @ K[t] - V[t], K[t])
        Oref[t] = W @ Q[t]
    assert np.abs(O - Oref).max() <= 1e-12
    assert np.abs(Wf - W).max() <= 1e-12


@pytest.mark.parametrize("C", [1, 4, 7, 19])
def test_inclusive_linear_ip_is_causal_linear_attention(C):
    """Linear net, inner-product loss: the gradient does not depend on W, so for
    every chunk size o_t = W0 q_t + step * sum_{s <= t} eta_s v_s (k_s . q_t):
    causal (token-inclusive) linear attention."""
    rng = np.random.default_rng(32)
    d, T, step = 6, 19, 0.7
    W0 = rng.standard_normal((d, d))
    Q, K, V = (rng.standard_normal((T, d)) for _ in range(3))
    eta = rng.uniform(0, 0.5, T)
    cfg = orc.OracleCfg(chunk=C, fast_net="linear", loss="ip", mode="inclusive", muon=False, wnorm=False,
                        step=step)
    O, (Wf,) = orc.ttt_head(cfg, Q, K, V, eta, (W0,))
    A = np.tril(Q @ K.T) * eta[None, :]
    Oref = Q @ W0.T + step * A @ V
    assert np.abs(O - Oref).max() <= 1e-12
    assert np.abs(Wf - (W0 + step * (eta[:, None] * V).T @ K)).max() <= 1e-12


def test_inclusive_chunk1_swiglu_is_the_per_token_recurrence():
    """SwiGLU net, MSE, chunks of one token: update with token t, then output
    with the updated weights, token after token."""
    rng = np.random.default_rng(33)
    d, dh, T = 4, 6, 9
    W = _rand_weights("swiglu", d, dh, rng)
    Q, K, V = (rng.standard_normal((T, d)) for _ in range(3))
    eta = rng.uniform(0, 0.3, T)
    cfg = orc.OracleCfg(chunk=1, loss="mse", mode="inclusive", muon=False, wnorm=False)
    O, Wf = orc.ttt_head(cfg, Q, K, V, eta, W)
    Wt = tuple(w.copy() for w in W)
    for t in range(T):
        g = orc.swiglu_grad(Wt, K[t:t + 1], V[t:t + 1], eta[t:t + 1], "mse")
        Wt = tuple(w - gj for w, gj in zip(Wt, g))
        assert np.abs(O[t] - orc.swiglu_apply(Wt, Q[t:t + 1])[0]).max() <= 1e-12
    for a, b in zip(Wf, Wt):
        assert np.abs(a - b).max() <= 1e-12


@pytest.mark.parametrize("loss", ["ip", "mse"])
def test_inclusive_swiglu_chunk_equals_its_dual_form(loss):
    """Each layer of the SwiGLU net is linear in its weights and each token's
    gradient is an outer product, so the prefix weights never need forming:
    A_q = Q W1^T - step tril(Q K^T) DA, B_q = Q W3^T - step tril(Q K^T) DB,
    H_q = silu(A_q) * B_q, O = H_q W2^T - step tril(H_q H_k^T) Yh, where DA,
    DB, H_k, Yh = eta * dl/df are the keys' quantities at the chunk's starting
    weights."""
    rng = np.random.default_rng(34)
    d, dh, C, step = 5, 8, 11, 0.6
    W1, W2, W3 = _rand_weights("swiglu", d, dh, rng)
    Q, K, V = (rng.standard_normal((C, d)) for _ in range(3))
    eta = rng.uniform(0, 0.4, C)
    cfg = orc.OracleCfg(chunk=C, loss=loss, mode="inclusive", muon=False, wnorm=False, step=step)
    got = orc.apply_inclusive(cfg, (W1, W2, W3), Q, K, V, eta)
    A, Bm = K @ W1.T, K @ W3.T
    sg = 1.0 / (1.0 + np.exp(-A))
    Hk = A * sg * Bm
    Y = (Hk @ W2.T - V) if loss == "mse" else -V
    Yh = eta[:, None] * Y
    DH = Yh @ W2
    DA = DH * Bm * sg * (1.0 + A * (1.0 - sg))
    DB = DH * A * sg
    L = np.tril(Q @ K.T)
    Aq = Q @ W1.T - step * L @ DA
    Bq = Q @ W3.T - step * L @ DB
    Hq = Aq / (1.0 + np.exp(-Aq)) * Bq
    Oref = Hq @ W2.T - step * np.tril(Hq @ Hk.T) @ Yh
    assert np.abs(got - Oref).max() <= 1e-12 * max(1.0, np.abs(Oref).max())


def test_inclusive_mode_refuses_chunk_level_optimisers():
    cfg = orc.OracleCfg(chunk=4, mode="inclusive", muon=True, wnorm=False)
    rng = np.random.default_rng(35)
    W = _rand_weights("swiglu", 4, 6, rng)
    X = rng.standard_normal((8, 4))
    with pytest.raises(ValueError):
        orc.ttt_head(cfg, X, X, X, np.ones(8), W)


def test_zero_rate_target_views_never_change_the_weights():
    """Novel-view synthesis (LaCT page §3.1): one chunk over a set of views in
    which the target views only query. Their tokens carry rate 0, so whatever
    their keys and values, the weights (and so every output) are those of the
    input views alone."""
    rng = np.random.default_rng(36)
    d, dh, T = 5, 8, 48
    W = _rand_weights("swiglu", d, dh, rng)
    Q, K, V = (rng.standard_normal((T, d)) for _ in range(3))
    target = (np.arange(T) // 6) % 4 == 3           # every fourth view of 6 tokens
    eta = np.where(target, 0.0, rng.uniform(0, 0.3, T))
    cfg = orc.OracleCfg(chunk=T, mode="single", muon=True, wnorm=True)
    O, Wf = orc.ttt_head(cfg, Q, K, V, eta, W)
    K2, V2 = K.copy(), V.copy()
    K2[target] = rng.standard_normal((int(target.sum()), d))
    V2[target] = rng.standard_normal((int(target.sum()), d))
    O2, Wf2 = orc.ttt_head(cfg, Q, K2, V2, eta, W)
    assert np.array_equal(O, O2)
    assert all(np.array_equal(a, b) for a, b in zip(Wf, Wf2))
    # and the input views alone give the same update
    keep = ~target
    cfg_in = orc.OracleCfg(chunk=int(keep.sum()), mode="single", muon=True, wnorm=True)
    _, Wf3 = orc.ttt_head(cfg_in, Q[keep], K[keep], V[keep], eta[keep], W)
    for a, b in zip(Wf, Wf3):
        assert np.abs(a - b).max() <= 1e-12


# ---------------------------------------------------------------- backward (outer loop)
@pytest.mark.parametrize("loss", ["mse", "ip"])
@pytest.mark.parametrize("C,mask", [(1, None), (4, None), (5, [1, 0, 1, 1])])
def test_linear_backward_matches_central_differences(loss, C, mask):
    """Every gradient of L = sum dO.O + sum dWf.Wf against central finite
    differences of the forward oracle (h = 1e-6), on a tiny head with a ragged
    last chunk."""
    rng = np.random.default_rng(41)
    d, T, step = 3, 17, 0.8
    W0 = rng.standard_normal((d, d)) / np.sqrt(d)
    Q, K, V = (rng.standard_normal((T, d)) for _ in range(3))
    lr = rng.uniform(0.05, 0.3, T)
    dO = rng.standard_normal((T, d))
    dWf = rng.standard_normal((d, d))
    cfg = orc.OracleCfg(chunk=C, fast_net="linear", loss=loss, muon=False, wnorm=False, step=step, mask=mask)

    def L(Q_, K_, V_, lr_, W_):
        O, (Wf,) = orc.ttt_head(cfg, Q_, K_, V_, lr_, (W_,))
        return float((dO * O).sum() + (dWf * Wf).sum())

    got = orc.linear_head_backward(cfg, Q, K, V, lr, W0, dO, dWf)
    args = [Q, K, V, lr, W0]
    h = 1e-6
    for i, g in enumerate(got):
        num = np.zeros_like(g)
        for idx in np.ndindex(*g.shape):
            up = [a.copy() for a in args]
            dn = [a.copy() for a in args]
            up[i][idx] += h
            dn[i][idx] -= h
            num[idx] = (L(*up) - L(*dn)) / (2 * h)
        assert np.abs(g - num).max() <= 1e-6 * max(1.0, np.abs(num).max()), (i, np.abs(g - num).max())


@pytest.mark.parametrize("loss", ["ip", "mse"])
@pytest.mark.parametrize("C,mask", [(3, None), (5, [1, 0, 1])])
def test_swiglu_backward_matches_central_differences(loss, C, mask):
    """The SwiGLU backward (automatic differentiation of an fp64 torch forward)
    against central finite differences of the NumPy forward oracle ttt_head:
    every input, a ragged last chunk, an update mask."""
    rng = np.random.default_rng(43)
    d, dh, T = 3, 4, 13
    step = 0.7 if loss == "ip" else 0.3  # MSE's inner loop diverges at larger steps
    W0 = _rand_weights("swiglu", d, dh, rng)
    Q, K, V = (rng.standard_normal((T, d)) for _ in range(3))
    lr = rng.uniform(0.05, 0.3, T)
    dO = rng.standard_normal((T, d))
    dWf = tuple(rng.standard_normal(w.shape) for w in W0)
    cfg = orc.OracleCfg(chunk=C, fast_net="swiglu", loss=loss, muon=False, wnorm=False, step=step, mask=mask)

    def L(Q_, K_, V_, lr_, W1_, W2_, W3_):
        O, Wf = orc.ttt_head(cfg, Q_, K_, V_, lr_, (W1_, W2_, W3_))
        return float((dO * O).sum() + sum((a * b).sum() for a, b in zip(dWf, Wf)))

    dQ, dK, dV, dlr, dW0 = orc.swiglu_head_backward(cfg, Q, K, V, lr, W0, dO, dWf)
    got = [dQ, dK, dV, dlr, *dW0]
    args = [Q, K, V, lr, *W0]
    h = 1e-6
    for i, g in enumerate(got):
        num = np.zeros_like(g)
        for idx in np.ndindex(*g.shape):
            up = [a.copy() for a in args]
            dn = [a.copy() for a in args]
            up[i][idx] += h
            dn[i][idx] -= h
            num[idx] = (L(*up) - L(*dn)) / (2 * h)
        assert np.abs(g - num).max() <= 1e-6 * max(1.0, np.abs(num).max()), (i, np.abs(g - num).max())
