"""Pins of the fp64 oracle against facts fixed outside the oracle itself:
hand-derived goldens, closed forms, independent library routines,
invariants of the mathematics and finite differences.  CPU only."""
import math
import os

import numpy as np
import pytest
import torch

import chain_synth as cs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
TIGHT = 1e-11


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b)) / max(1e-300, np.max(np.abs(b))))


def f64(*xs):
    return [torch.as_tensor(x).to(torch.float64) for x in xs]


# ----------------------------------------------------------------- goldens
def test_golden_two_keys(orc):
    lines = [l.split() for l in open(os.path.join(GOLDEN, "attn_two_keys.txt"))
             if l.strip() and not l.startswith("#")]
    vec = {l[0]: [float(x) for x in l[1:]] for l in lines if l[0] in "qkv"}
    Q = torch.tensor(vec["q"], dtype=torch.float64).reshape(1, 2, 1)
    K = torch.tensor(vec["k"], dtype=torch.float64).reshape(1, 2, 1)
    V = torch.tensor(vec["v"], dtype=torch.float64).reshape(1, 2, 1)
    rows = [l for l in lines if l[0] not in "qkv"]
    assert len(rows) == 4
    for causal in (0, 1):
        O, L = orc.softmax_fwd(Q, K, V, 1.0, bool(causal))
        for c, i, o, lse in rows:
            if int(c) != causal:
                continue
            assert abs(O[0, int(i), 0] - float(o)) < 1e-14
            assert abs(L[0, int(i)] - float(lse)) < 1e-14


def test_golden_identity_chain(orc):
    m = {}
    for l in open(os.path.join(GOLDEN, "identity_chain_2x2.txt")):
        if l.strip() and not l.startswith("#"):
            t = l.split()
            r, c = int(t[1]), int(t[2])
            m[t[0]] = np.array([float(x) for x in t[3:]]).reshape(r, c)
    O = orc.chain_fwd(m["A"], m["B"], m["C"], orc.F_IDENTITY)
    assert np.array_equal(O, m["O"])


# -------------------------------------------------------------- closed forms
@pytest.mark.parametrize("causal", [False, True])
def test_uniform_scores(orc, causal):
    # Q = 0 makes every score 0: P is uniform over the allowed keys, so
    # O_i is the mean of V over them and LSE_i = ln(#keys).
    n, d = 37, 5
    Q = torch.zeros(2, n, d, dtype=torch.float64)
    K = cs.normal((2, n, d), seed=101, dtype=torch.float64)
    V = cs.normal((2, n, 3), seed=102, dtype=torch.float64)
    O, L = orc.softmax_fwd(Q, K, V, 0.3, causal)
    for i in range(n):
        cnt = i + 1 if causal else n
        assert np.allclose(O[:, i], V[:, :cnt].mean(1).numpy(), rtol=0, atol=1e-13)
        assert abs(L[0, i] - math.log(cnt)) < 1e-13


def test_causal_row_zero(orc):
    n, d = 19, 7
    Q, K, V = cs.attn_inputs(3, n, d, seed=11, dtype=torch.float32)
    O, L = orc.softmax_fwd(Q, K, V, 0.25, True)
    q0 = Q[:, 0].double()
    k0 = K[:, 0].double()
    assert np.array_equal(O[:, 0], V[:, 0].double().numpy())
    assert np.allclose(L[:, 0], (0.25 * (q0 * k0).sum(-1)).numpy(), rtol=1e-15, atol=1e-15)


def test_rows_sum_to_one(orc):
    # C = all ones: O = sum_j P_ij = 1 for every row.
    Q, K, _ = cs.attn_inputs(2, 50, 8, seed=5, dtype=torch.float32)
    V = torch.ones(2, 50, 4)
    for causal in (False, True):
        O, _ = orc.softmax_fwd(Q, K, V, 0.7, causal)
        assert np.max(np.abs(O - 1.0)) < 1e-14


def test_shift_invariance_and_large_scores(orc):
    # Adding c to every score of a row (an extra feature: K[:, d] = 1,
    # Q[i, d] = c / scale) leaves O unchanged and adds c to LSE; huge scores
    # produce no inf/NaN.
    n, d, scale = 24, 6, 0.5
    Q, K, V = f64(*cs.attn_inputs(1, n, d, seed=7, dtype=torch.float32))
    shift = torch.linspace(-800.0, 900.0, n, dtype=torch.float64)
    Qa = torch.cat([Q, (shift / scale).reshape(1, n, 1)], -1)
    Ka = torch.cat([K, torch.ones(1, n, 1, dtype=torch.float64)], -1)
    for causal in (False, True):
        O0, L0 = orc.softmax_fwd(Q, K, V, scale, causal)
        O1, L1 = orc.softmax_fwd(Qa, Ka, V, scale, causal)
        assert np.all(np.isfinite(O1)) and np.all(np.isfinite(L1))
        assert rel(O1, O0) < 1e-12
        assert np.allclose(L1 - L0, shift.numpy().reshape(1, n), rtol=0, atol=1e-10)


def test_one_hot_hard_attention(orc):
    # Keys are scaled one-hot vectors, queries one-hot: each row attends to
    # exactly one key, so O is a row permutation of V.
    n = d = 16
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(3))
    K = torch.zeros(1, n, d, dtype=torch.float64)
    K[0, torch.arange(n), perm] = 1.0
    Q = torch.zeros(1, n, d, dtype=torch.float64)
    tgt = torch.randperm(n, generator=torch.Generator().manual_seed(4))
    Q[0, torch.arange(n), perm[tgt]] = 1.0
    V = cs.normal((1, n, 5), seed=103, dtype=torch.float64)
    O, _ = orc.softmax_fwd(Q, K, V, 2000.0, False)
    assert np.allclose(O[0], V[0, tgt].numpy(), rtol=0, atol=1e-12)


# ------------------------------------------------------ independent library
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,d", [(64, 16), (33, 8)])
def test_fwd_vs_sdpa(orc, causal, n, d):
    Q, K, V = f64(*cs.attn_inputs(3, n, d, seed=21, dtype=torch.float32))
    scale = 1.0 / math.sqrt(d)
    ref = torch.nn.functional.scaled_dot_product_attention(
        Q, K, V, is_causal=causal, scale=scale)
    O, _ = orc.softmax_fwd(Q, K, V, scale, causal)
    assert rel(O, ref.numpy()) < TIGHT


def test_fwd_bf16_inputs_widen_exactly(orc):
    Q, K, V = cs.attn_inputs(2, 40, 8, seed=9, dtype=torch.bfloat16)
    O1, L1 = orc.softmax_fwd(Q, K, V, 0.3, True)
    O2, L2 = orc.softmax_fwd(Q.double(), K.double(), V.double(), 0.3, True)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_fwd_sampled_rows_match_full(orc):
    Q, K, V = cs.attn_inputs(3, 70, 8, seed=13, dtype=torch.bfloat16)
    O, L = orc.softmax_fwd(Q, K, V, 0.4, True)
    rows = cs.sample_rows(3, 70, 6, seed=1)
    Os, Ls = orc.softmax_fwd(Q, K, V, 0.4, True, rows=rows)
    r = rows.numpy()
    assert np.array_equal(Os, O[r[:, 0], r[:, 1]])
    assert np.array_equal(Ls, L[r[:, 0], r[:, 1]])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("p", [2, 4])
def test_block_merge_equals_unblocked(orc, causal, p):
    Q, K, V = cs.attn_inputs(2, 48, 8, seed=17, dtype=torch.float32)
    O, L = orc.softmax_fwd(Q, K, V, 0.35, causal)
    Ob, Lb = orc.softmax_fwd_blocked(Q, K, V, 0.35, causal, p, p)
    assert rel(Ob, O) < 1e-12
    assert rel(Lb, L) < 1e-12


# ------------------------------------------------------------------ backward
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_vs_autograd(orc, causal):
    n, d = 40, 8
    Q, K, V, G = f64(*cs.attn_inputs(2, n, d, seed=31, dtype=torch.float32, with_do=True))
    scale = 1.0 / math.sqrt(d)
    q, k, v = (t.clone().requires_grad_() for t in (Q, K, V))
    out = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale)
    out.backward(G)
    dQ, dK, dV, D = orc.softmax_bwd(Q, K, V, G, scale, causal)
    assert rel(dQ, q.grad.numpy()) < TIGHT
    assert rel(dK, k.grad.numpy()) < TIGHT
    assert rel(dV, v.grad.numpy()) < TIGHT
    # D_i = sum_e dO_ie O_ie equals sum_j P_ij dP_ij
    assert rel(D, (G * out.detach()).sum(-1).numpy()) < TIGHT


def test_bwd_finite_differences(orc):
    # Central differences of L = sum(O * G) through the oracle's forward.
    n, d = 6, 3
    Q, K, V, G = f64(*cs.attn_inputs(1, n, d, seed=41, dtype=torch.float32, with_do=True))
    scale = 0.8
    dQ, dK, dV, _ = orc.softmax_bwd(Q, K, V, G, scale, True)
    h = 1e-6

    def loss(q, k, v):
        O, _ = orc.softmax_fwd(q, k, v, scale, True)
        return float((O * G.numpy()).sum())

    for name, T, grad in (("Q", Q, dQ), ("K", K, dK), ("V", V, dV)):
        num = np.zeros_like(grad)
        for idx in np.ndindex(*T.shape):
            tp, tm = T.clone(), T.clone()
            tp[idx] += h
            tm[idx] -= h
            args_p = {"Q": Q, "K": K, "V": V}
            args_m = dict(args_p)
            args_p[name], args_m[name] = tp, tm
            num[idx] = (loss(args_p["Q"], args_p["K"], args_p["V"])
                        - loss(args_m["Q"], args_m["K"], args_m["V"])) / (2 * h)
        assert rel(grad, num) < 1e-7, name


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_invariants(orc, causal):
    Q, K, V, G = cs.attn_inputs(2, 64, 16, seed=51, dtype=torch.bfloat16, with_do=True)
    dQ, dK, dV, _ = orc.softmax_bwd(Q, K, V, G, 0.25, causal)
    # rows of dS sum to zero, so the key-sum of dK vanishes
    assert np.max(np.abs(dK.sum(1))) < 1e-10 * np.max(np.abs(dK))
    # rows of P sum to one, so the key-sum of dV equals the row-sum of dO
    assert np.allclose(dV.sum(1), G.double().sum(1).numpy(), rtol=0, atol=1e-11)


def test_bwd_row_and_column_ranges(orc):
    # With causal masking the key columns j >= i0 receive contributions only
    # from rows i >= j, so rows [i0, n) give them exactly.
    n = 50
    Q, K, V, G = cs.attn_inputs(3, n, 8, seed=61, dtype=torch.float32, with_do=True)
    dQ, dK, dV, D = orc.softmax_bwd(Q, K, V, G, 0.3, True)
    i0 = 37
    dQp, dKp, dVp, Dp = orc.softmax_bwd(Q, K, V, G, 0.3, True, heads=(1, 3),
                                        row_range=(i0, n), col_range=(i0, n))
    assert rel(dQp, dQ[1:3, i0:]) < 1e-14
    assert rel(Dp, D[1:3, i0:]) < 1e-14
    assert rel(dKp, dK[1:3, i0:]) < 1e-12
    assert rel(dVp, dV[1:3, i0:]) < 1e-12


def test_bwd_repeatable_and_key_block_of_full_rows(orc):
    # Repeated calls give identical bits (each thread's share of the dK, dV
    # row sums is fixed and the shares are added in thread order), and a key
    # block taken over every row equals the same block of the full gradient:
    # the form the full-length parity tests use.
    n = 300
    Q, K, V, G = cs.attn_inputs(2, n, 16, seed=63, dtype=torch.bfloat16, with_do=True)
    a = orc.softmax_bwd(Q, K, V, G, 0.25, True, heads=(1, 2), row_range=(0, n), col_range=(0, 128))
    b = orc.softmax_bwd(Q, K, V, G, 0.25, True, heads=(1, 2), row_range=(0, n), col_range=(0, 128))
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    dQ, dK, dV, _ = orc.softmax_bwd(Q, K, V, G, 0.25, True)
    assert rel(a[0], dQ[1:2]) < 1e-14
    assert rel(a[1], dK[1:2, :128]) < 1e-12
    assert rel(a[2], dV[1:2, :128]) < 1e-12


# --------------------------------------------------------------------- chain
def test_identity_chain_associativity(orc):
    A, B, C = (np.random.default_rng(s).standard_normal(sh)
               for s, sh in ((1, (23, 17)), (2, (17, 29)), (3, (29, 11))))
    O = orc.chain_fwd(A, B, C, orc.F_IDENTITY)
    assert rel(O, A @ (B @ C)) < 1e-12


def test_gelu_chain_vs_library(orc):
    A, B = (np.random.default_rng(s).standard_normal(sh) * 2
            for s, sh in ((4, (9, 13)), (5, (13, 21))))
    I = np.eye(21)
    O = orc.chain_fwd(A, B, I, orc.F_GELU_TANH)
    ref = torch.nn.functional.gelu(torch.from_numpy(A @ B), approximate="tanh").numpy()
    assert rel(O, ref) < 1e-12
    # full chain against the library activation followed by a product
    C = np.random.default_rng(6).standard_normal((21, 7))
    O2 = orc.chain_fwd(A, B, C, orc.F_GELU_TANH)
    assert rel(O2, ref @ C) < 1e-12


def test_gelu_properties(orc):
    t = np.array([[0.0, 1e-3, 0.5, -0.5, 3.0, -3.0, 12.0, -12.0, 40.0, -40.0]])
    g = orc.chain_fwd(t.T.copy(), np.ones((1, 1)), np.ones((1, 1)), orc.F_GELU_TANH)[:, 0]
    gn = orc.chain_fwd(-t.T.copy(), np.ones((1, 1)), np.ones((1, 1)), orc.F_GELU_TANH)[:, 0]
    assert g[0] == 0.0
    assert np.allclose(g - gn, t[0], rtol=0, atol=1e-14)  # odd part is x
    assert abs(g[8] - 40.0) < 1e-12 and abs(g[9]) < 1e-12  # asymptotes
    assert abs(g[6] - 12.0) < 1e-12


def test_softmax_chain_matches_attention(orc):
    # f = softmax in the general chain with B = K^T reproduces attention.
    Q, K, V = f64(*cs.attn_inputs(1, 30, 6, seed=71, dtype=torch.float32))
    O, _ = orc.softmax_fwd(Q, K, V, 0.45, False)
    Oc = orc.chain_fwd(Q[0].numpy(), K[0].T.contiguous().numpy(), V[0].numpy(),
                       orc.F_SOFTMAX, 0.45)
    ref = torch.softmax(0.45 * Q[0] @ K[0].T, -1) @ V[0]
    assert rel(Oc, ref.numpy()) < TIGHT
    assert rel(O[0], Oc) < TIGHT


def test_chain_sampled_rows(orc):
    A, B, C = cs.mlp_inputs(40, 16, 24, 8, seed=81)
    O = orc.chain_fwd(A, B, C, orc.F_GELU_TANH)
    rows = [0, 5, 39, 17]
    Os = orc.chain_fwd(A, B, C, orc.F_GELU_TANH, rows=rows)
    assert np.array_equal(Os, O[rows])


# ------------------------------------------------------------ chain backward
def _chain_loss(orc, A, B, C, G, f):
    return float((orc.chain_fwd(A, B, C, f) * G).sum())


@pytest.mark.parametrize("f", ["gelu", "identity"])
def test_chain_bwd_finite_differences(orc, f):
    # Central differences of L = sum(O * G) through the oracle's forward.
    fc = orc.F_GELU_TANH if f == "gelu" else orc.F_IDENTITY
    rng = np.random.default_rng(91)
    A, B, C, G = (rng.standard_normal(sh) for sh in ((3, 4), (4, 5), (5, 2), (3, 2)))
    dA, dBc, dC = orc.chain_bwd(A, B, C, G, fc)
    h = 1e-6
    for name, X, grad in (("A", A, dA), ("B", B, dBc.T), ("C", C, dC)):
        num = np.zeros_like(X)
        for idx in np.ndindex(*X.shape):
            xp, xm = X.copy(), X.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"A": A, "B": B, "C": C}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            num[idx] = (_chain_loss(orc, args_p["A"], args_p["B"], args_p["C"], G, fc)
                        - _chain_loss(orc, args_m["A"], args_m["B"], args_m["C"], G, fc)) / (2 * h)
        assert rel(grad, num) < 1e-7, (f, name)


def test_chain_bwd_identity_closed_form(orc):
    # f = identity: dA = G C^T B^T, dB = A^T G C^T, dC = (A B)^T G.
    rng = np.random.default_rng(92)
    A, B, C, G = (rng.standard_normal(sh) for sh in ((19, 11), (11, 23), (23, 7), (19, 7)))
    dA, dBc, dC = orc.chain_bwd(A, B, C, G, orc.F_IDENTITY)
    assert rel(dA, G @ C.T @ B.T) < 1e-12
    assert rel(dBc.T, A.T @ G @ C.T) < 1e-12
    assert rel(dC, (A @ B).T @ G) < 1e-12


def test_chain_bwd_vs_autograd(orc):
    # fp64 autograd of the library's tanh GeLU, an independent derivative.
    rng = np.random.default_rng(93)
    A, B, C, G = (torch.from_numpy(rng.standard_normal(sh) * sc)
                  for sh, sc in (((17, 9), 1.0), ((9, 31), 0.7), ((31, 5), 0.4), ((17, 5), 1.0)))
    A.requires_grad_(True)
    B.requires_grad_(True)
    C.requires_grad_(True)
    O = torch.nn.functional.gelu(A @ B, approximate="tanh") @ C
    (O * G).sum().backward()
    dA, dBc, dC = orc.chain_bwd(A.detach(), B.detach(), C.detach(), G, orc.F_GELU_TANH)
    assert rel(dA, A.grad.numpy()) < 1e-12
    assert rel(dBc.T, B.grad.numpy()) < 1e-12
    assert rel(dC, C.grad.numpy()) < 1e-12


def test_gelu_grad_symmetry(orc):
    # gelu(x) - gelu(-x) = x, so gelu'(x) + gelu'(-x) = 1; gelu'(0) = 1/2.
    one = np.ones((1, 1))
    for t in (0.0, 0.3, -1.7, 2.5, 6.0):
        g = lambda x: orc.chain_bwd(np.array([[x]]), one, one, one, orc.F_GELU_TANH)[0][0, 0]
        assert abs(g(t) + g(-t) - 1.0) < 1e-14, t
    assert abs(orc.chain_bwd(np.zeros((1, 1)), one, one, one, orc.F_GELU_TANH)[0][0, 0] - 0.5) < 1e-15


def test_chain_bwd_sampled_match_full(orc):
    A, B, C = cs.mlp_inputs(40, 16, 24, 8, seed=94)
    G = cs.normal((40, 8), seed=95)
    dA, dB, dC = orc.chain_bwd(A, B, C, G, orc.F_GELU_TANH)
    rows, hid = [0, 7, 39], [1, 23, 10]
    sA, sB, sC = orc.chain_bwd(A, B, C, G, orc.F_GELU_TANH, rows=rows, hidden=hid)
    assert np.array_equal(sA, dA[rows]) and np.array_equal(sB, dB[hid]) and np.array_equal(sC, dC[hid])


# ------------------------------------------------------------------ relayout
@pytest.mark.parametrize("p,n_loc,H,d,g", [(4, 5, 8, 3, 0), (4, 5, 8, 3, 3), (2, 7, 6, 4, 1)])
def test_relayout_vs_transpose(orc, p, n_loc, H, d, g):
    x = cs.iota16((p, n_loc, H, d))
    out, shape = orc.relayout(x, p, g)
    Hl = H // p
    ref = (x.numpy().reshape(p, n_loc, p, Hl, d)[:, :, g]  # [p][n_loc][Hl][d]
           .transpose(2, 0, 1, 3).reshape(Hl, p * n_loc, d))
    assert shape == (Hl, p * n_loc, d)
    assert np.array_equal(out.view(np.int16).reshape(shape), ref)


def test_relayout_round_trip(orc):
    p, n_loc, H, d = 4, 6, 8, 5
    x = cs.normal((p, n_loc, H, d), seed=91)
    back = np.zeros(x.numel() * 2, np.uint8)
    for g in range(p):
        out, shape = orc.relayout(x, p, g)
        orc.relayout_inverse(torch.from_numpy(out.view(np.int16).reshape(shape)), p, n_loc, H,
                             g, into=back)
    assert np.array_equal(back, x.view(torch.uint8).numpy().reshape(-1))


# ------------------------------------------------------------ e4m3 inputs
def test_e4m3_decode_closed_forms(orc):
    # values the format fixes: sign, 4 exponent bits with bias 7, 3 mantissa
    # bits, exponent field 0 subnormal, S.1111.111 NaN
    cases = {0x00: 0.0, 0x38: 1.0, 0x40: 2.0, 0x3C: 1.5, 0xB8: -1.0, 0x30: 0.5,
             0x7E: 448.0, 0xFE: -448.0, 0x77: 240.0, 0x08: 2.0 ** -6, 0x01: 2.0 ** -9,
             0x07: 7 * 2.0 ** -9, 0x81: -(2.0 ** -9)}
    codes = np.array(list(cases), dtype=np.uint8)
    got = orc.e4m3_decode(codes)
    assert list(got) == [cases[int(c)] for c in codes]
    assert np.isnan(orc.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()


def test_e4m3_decode_matches_torch(orc):
    # every code against the library's float8_e4m3fn conversion
    codes = np.arange(256, dtype=np.uint8)
    ours = orc.e4m3_decode(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float32).double().numpy()
    nan = np.isnan(ref)
    assert set(np.flatnonzero(nan).tolist()) == {0x7F, 0xFF}
    np.testing.assert_array_equal(np.isnan(ours), nan)
    np.testing.assert_array_equal(ours[~nan], ref[~nan])


def test_e4m3_decode_monotone_and_odd(orc):
    pos = orc.e4m3_decode(np.arange(0x00, 0x7F, dtype=np.uint8))
    neg = orc.e4m3_decode(np.arange(0x80, 0xFF, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)
    np.testing.assert_array_equal(neg, -pos)


def test_oracle_softmax_on_e4m3_codes(orc):
    # the oracle fed e4m3 codes computes on their exact values: identical to
    # feeding those values in fp64, and to the library's scaled-dot-product
    # attention on them
    q, k, v = cs.attn_inputs(2, 40, 8, seed=61, dtype=torch.float8_e4m3fn)
    O8, L8 = orc.softmax_fwd(q, k, v, 0.3, True)
    dec = [torch.from_numpy(orc.e4m3_decode(x)) for x in (q, k, v)]
    O64, L64 = orc.softmax_fwd(*dec, 0.3, True)
    np.testing.assert_array_equal(O8, O64)
    np.testing.assert_array_equal(L8, L64)
    ref = torch.nn.functional.scaled_dot_product_attention(*dec, is_causal=True, scale=0.3)
    assert rel(O8, ref.numpy()) < TIGHT
