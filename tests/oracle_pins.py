"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Every check takes a loaded oracle library (``oracle.load_library()`` or a
mutated build of the same source) and raises AssertionError when the oracle
disagrees with what the mathematics fixes.  ``tests/test_oracle_pins.py`` runs
them on the real oracle; ``tests/test_oracle_mutants.py`` runs them on copies
of the oracle with a planted mistake and requires at least one to fail.

Kinds of pin (the pages print no worked attention example with values):
  * brute force at 50 significant digits with Python's ``decimal`` on tiny
    inputs, without the max subtraction the oracle uses;
  * a library routine: scipy's softmax / logsumexp on the masked score matrix;
  * closed forms (Q = 0, row 0, two keys, constant V, V = identity);
  * invariants (key shift, joint key/value permutation, prefix equivalence,
    scale folding, decode = last causal row);
  * one count printed on the page "Hand-written masked multi-head attention
    CUDA kernel" section 1 (the causal mask of a 2048-token sequence keeps
    about 2.09 million of about 4.19 million scores), in tests/golden/.
"""
from __future__ import annotations

import decimal
import json
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _small_grid(rng, shape, denom=8, lo=-12, hi=12):
    """Values k/denom with small integers k: exact in float32, sums exact too."""
    return (rng.integers(lo, hi + 1, size=shape) / denom).astype(np.float32)


def _decimal_attention(Q, K, V, scale, causal, key_lens=None):
    """Brute force: full masked score matrix, exp without max shift, 50 digits.
    With ``key_lens`` keys j >= key_lens[b] are masked too; a row with no valid
    key gets O = 0 and LSE = -inf (the empty sum)."""
    ctx = decimal.Context(prec=50)
    Dm = lambda x: ctx.create_decimal_from_float(float(x))
    B, H, S, D = Q.shape
    O = np.zeros((B, H, S, D))
    L = np.zeros((B, H, S))
    sc = Dm(scale)
    for b in range(B):
        for h in range(H):
            for i in range(S):
                w = []
                for j in range(S):
                    if (causal and j > i) or (key_lens is not None and j >= key_lens[b]):
                        w.append(ctx.create_decimal(0))  # exp(-inf)
                        continue
                    dot = sum((Dm(Q[b, h, i, d]) * Dm(K[b, h, j, d]) for d in range(D)),
                              ctx.create_decimal(0))
                    w.append(ctx.exp(ctx.multiply(sc, dot)))
                Z = sum(w, ctx.create_decimal(0))
                if Z == 0:
                    O[b, h, i, :] = 0.0
                    L[b, h, i] = -math.inf
                    continue
                for d in range(D):
                    num = sum((w[j] * Dm(V[b, h, j, d]) for j in range(S)), ctx.create_decimal(0))
                    O[b, h, i, d] = float(ctx.divide(num, Z))
                L[b, h, i] = float(ctx.ln(Z))
    return O, L


def check_bruteforce_decimal(lib):
    rng = np.random.default_rng(7)
    for causal in (True, False):
        for (B, H, S, D) in ((1, 2, 5, 3), (2, 1, 7, 4), (1, 1, 1, 2)):
            Q = rng.standard_normal((B, H, S, D)).astype(np.float32)
            K = rng.standard_normal((B, H, S, D)).astype(np.float32)
            V = rng.standard_normal((B, H, S, D)).astype(np.float32)
            scale = 0.7
            O, L = oracle.attention(Q, K, V, scale, causal, lib=lib)
            Ob, Lb = _decimal_attention(Q, K, V, scale, causal)
            assert np.max(np.abs(O - Ob)) <= 1e-13, ("O", causal, (B, H, S, D))
            assert np.max(np.abs(L - Lb)) <= 1e-13, ("LSE", causal, (B, H, S, D))


def check_library_softmax(lib):
    from scipy.special import logsumexp, softmax
    rng = np.random.default_rng(11)
    B, H, S, D = 2, 3, 37, 16
    Q = (3 * rng.standard_normal((B, H, S, D))).astype(np.float32)
    K = (3 * rng.standard_normal((B, H, S, D))).astype(np.float32)
    V = rng.standard_normal((B, H, S, D)).astype(np.float32)
    scale = 1 / math.sqrt(D)
    for causal in (True, False):
        O, L = oracle.attention(Q, K, V, scale, causal, lib=lib)
        s = scale * np.einsum("bhid,bhjd->bhij", Q.astype(np.float64), K.astype(np.float64))
        if causal:
            s = np.where(np.tril(np.ones((S, S), dtype=bool)), s, -np.inf)
        P = softmax(s, axis=-1)
        Oref = P @ V.astype(np.float64)
        Lref = logsumexp(s, axis=-1)
        assert np.max(np.abs(O - Oref)) <= 1e-12, causal
        assert np.max(np.abs(L - Lref)) <= 1e-12, causal


def check_zero_query_prefix_mean(lib):
    rng = np.random.default_rng(3)
    B, H, S, D = 1, 2, 19, 5
    Q = np.zeros((B, H, S, D), np.float32)
    K = rng.standard_normal((B, H, S, D)).astype(np.float32)
    V = rng.standard_normal((B, H, S, D)).astype(np.float32)
    O, L = oracle.attention(Q, K, V, 0.5, True, lib=lib)
    counts = np.arange(1, S + 1, dtype=np.float64)
    prefix_mean = np.cumsum(V.astype(np.float64), axis=2) / counts[None, None, :, None]
    assert np.max(np.abs(O - prefix_mean)) <= 1e-14
    assert np.max(np.abs(L - np.log(counts)[None, None, :])) <= 1e-14
    O, L = oracle.attention(Q, K, V, 0.5, False, lib=lib)
    full_mean = V.astype(np.float64).mean(axis=2, keepdims=True)
    assert np.max(np.abs(O - full_mean)) <= 1e-14
    assert np.max(np.abs(L - math.log(S))) <= 1e-14


def check_row0_and_two_keys(lib):
    rng = np.random.default_rng(5)
    B, H, S, D = 2, 2, 9, 6
    Q = rng.standard_normal((B, H, S, D)).astype(np.float32)
    K = rng.standard_normal((B, H, S, D)).astype(np.float32)
    V = rng.standard_normal((B, H, S, D)).astype(np.float32)
    scale = 0.37
    O, L = oracle.attention(Q, K, V, scale, True, lib=lib)
    for b in range(B):
        for h in range(H):
            q0k0 = math.fsum(float(Q[b, h, 0, d]) * float(K[b, h, 0, d]) for d in range(D))
            # row 0 sees only key 0: weight 1, so O_0 = V_0 and LSE_0 = its score
            assert np.max(np.abs(O[b, h, 0] - V[b, h, 0])) <= 1e-15
            assert abs(L[b, h, 0] - scale * q0k0) <= 1e-14
            # row 1 sees keys 0 and 1: logistic weights
            s0 = scale * math.fsum(float(Q[b, h, 1, d]) * float(K[b, h, 0, d]) for d in range(D))
            s1 = scale * math.fsum(float(Q[b, h, 1, d]) * float(K[b, h, 1, d]) for d in range(D))
            a0 = 1.0 / (1.0 + math.exp(s1 - s0))
            a1 = 1.0 / (1.0 + math.exp(s0 - s1))
            o1 = a0 * V[b, h, 0].astype(np.float64) + a1 * V[b, h, 1].astype(np.float64)
            assert np.max(np.abs(O[b, h, 1] - o1)) <= 1e-14
            lse1 = max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1)))
            assert abs(L[b, h, 1] - lse1) <= 1e-14


def check_constant_v(lib):
    rng = np.random.default_rng(9)
    B, H, S, D = 1, 3, 23, 4
    Q = (4 * rng.standard_normal((B, H, S, D))).astype(np.float32)
    K = (4 * rng.standard_normal((B, H, S, D))).astype(np.float32)
    V = np.full((B, H, S, D), -1.625, np.float32)
    for causal in (True, False):
        O, _ = oracle.attention(Q, K, V, 0.5, causal, lib=lib)
        assert np.max(np.abs(O + 1.625)) <= 1e-14


def check_identity_values_give_probabilities(lib):
    """With D = S and V = I, row i of O is row i of the attention matrix."""
    rng = np.random.default_rng(13)
    S = 12
    Q = rng.standard_normal((1, 1, S, S)).astype(np.float32)
    K = rng.standard_normal((1, 1, S, S)).astype(np.float32)
    V = np.eye(S, dtype=np.float32)[None, None]
    scale = 0.8
    for causal in (True, False):
        O, _ = oracle.attention(Q, K, V, scale, causal, lib=lib)
        P = O[0, 0]
        assert np.all(P >= 0)
        assert np.max(np.abs(P.sum(axis=1) - 1.0)) <= 1e-14
        if causal:
            assert np.all(P[np.triu_indices(S, 1)] == 0.0)   # above diagonal: excluded
            assert np.all(np.diag(P) > 0)                     # diagonal: included
        for i in range(S):
            n = i + 1 if causal else S
            s = [scale * math.fsum(float(Q[0, 0, i, d]) * float(K[0, 0, j, d]) for d in range(S))
                 for j in range(n)]
            for j in range(1, n):
                # ratio of two weights is exp of the score difference
                assert abs(math.log(P[i, j] / P[i, 0]) - (s[j] - s[0])) <= 1e-12


def check_key_shift_invariance(lib):
    rng = np.random.default_rng(17)
    B, H, S, D = 1, 2, 16, 8
    Q = _small_grid(rng, (B, H, S, D))
    K = _small_grid(rng, (B, H, S, D))
    V = rng.standard_normal((B, H, S, D)).astype(np.float32)
    w = _small_grid(rng, (D,))
    scale = 0.25
    for causal in (True, False):
        O1, L1 = oracle.attention(Q, K, V, scale, causal, lib=lib)
        O2, L2 = oracle.attention(Q, K + w[None, None, None, :], V, scale, causal, lib=lib)
        qw = scale * (Q.astype(np.float64) @ w.astype(np.float64))
        assert np.max(np.abs(O1 - O2)) <= 1e-13
        assert np.max(np.abs((L2 - L1) - qw)) <= 1e-12


def check_joint_permutation(lib):
    rng = np.random.default_rng(19)
    B, H, S, D = 2, 2, 21, 8
    Q = rng.standard_normal((B, H, S, D)).astype(np.float32)
    K = rng.standard_normal((B, H, S, D)).astype(np.float32)
    V = rng.standard_normal((B, H, S, D)).astype(np.float32)
    perm = rng.permutation(S)
    O1, L1 = oracle.attention(Q, K, V, 0.3, False, lib=lib)
    O2, L2 = oracle.attention(Q, K[:, :, perm], V[:, :, perm], 0.3, False, lib=lib)
    assert np.max(np.abs(O1 - O2)) <= 1e-13
    assert np.max(np.abs(L1 - L2)) <= 1e-13


def check_causal_row_is_prefix_attention(lib):
    rng = np.random.default_rng(23)
    B, H, S, D = 1, 1, 14, 6
    Q = rng.standard_normal((B, H, S, D)).astype(np.float32)
    K = rng.standard_normal((B, H, S, D)).astype(np.float32)
    V = rng.standard_normal((B, H, S, D)).astype(np.float32)
    Oc, Lc = oracle.attention(Q, K, V, 0.45, True, lib=lib)
    for i in range(S):
        On, Ln = oracle.attention(Q[:, :, :i + 1], K[:, :, :i + 1], V[:, :, :i + 1], 0.45, False,
                                  lib=lib)
        assert np.max(np.abs(Oc[0, 0, i] - On[0, 0, i])) <= 1e-15
        assert abs(Lc[0, 0, i] - Ln[0, 0, i]) <= 1e-15


def check_scale_folding(lib):
    rng = np.random.default_rng(29)
    B, H, S, D = 1, 2, 10, 4
    Q = rng.standard_normal((B, H, S, D)).astype(np.float32)
    K = rng.standard_normal((B, H, S, D)).astype(np.float32)
    V = rng.standard_normal((B, H, S, D)).astype(np.float32)
    O1, L1 = oracle.attention(Q, K, V, 0.5, True, lib=lib)
    O2, L2 = oracle.attention(Q * np.float32(2), K, V, 0.25, True, lib=lib)
    assert np.max(np.abs(O1 - O2)) <= 1e-14 and np.max(np.abs(L1 - L2)) <= 1e-14


def check_rows_subset(lib):
    rng = np.random.default_rng(31)
    B, H, S, D = 2, 3, 11, 5
    Q = rng.standard_normal((B, H, S, D)).astype(np.float32)
    K = rng.standard_normal((B, H, S, D)).astype(np.float32)
    V = rng.standard_normal((B, H, S, D)).astype(np.float32)
    O, L = oracle.attention(Q, K, V, 0.6, True, lib=lib)
    rows = np.array([0, 5, 10, 11, 33, 65, 40, 7])
    Or, Lr = oracle.attention(Q, K, V, 0.6, True, rows=rows, lib=lib)
    assert np.array_equal(Or, O.reshape(-1, D)[rows])
    assert np.array_equal(Lr, L.reshape(-1)[rows])
    # thread count does not change a single bit (each row is one thread's loop)
    O1, L1 = oracle.attention(Q, K, V, 0.6, True, nthreads=1, lib=lib)
    O4, L4 = oracle.attention(Q, K, V, 0.6, True, nthreads=4, lib=lib)
    assert np.array_equal(O1, O4) and np.array_equal(L1, L4)


def check_decode_is_last_causal_row(lib):
    rng = np.random.default_rng(37)
    H, D = 3, 8
    seqlens = np.array([5, 1, 9, 3], np.int32)
    B = seqlens.size
    seqs_k = [rng.standard_normal((int(L), H, D)).astype(np.float32) for L in seqlens]
    seqs_v = [rng.standard_normal((int(L), H, D)).astype(np.float32) for L in seqlens]
    q = rng.standard_normal((B, H, D)).astype(np.float32)
    Kc = np.concatenate(seqs_k)
    Vc = np.concatenate(seqs_v)
    Od, Ld = oracle.decode(q, Kc, Vc, seqlens, 0.4, lib=lib)
    for b, L in enumerate(seqlens):
        L = int(L)
        Kp = np.transpose(seqs_k[b], (1, 0, 2))[None]   # [1, H, L, D]
        Vp = np.transpose(seqs_v[b], (1, 0, 2))[None]
        Qp = np.zeros_like(Kp)
        Qp[0, :, L - 1] = q[b]
        Op, Lp = oracle.attention(Qp, Kp, Vp, 0.4, True, lib=lib)
        assert np.max(np.abs(Od[b] - Op[0, :, L - 1])) <= 1e-15
        assert np.max(np.abs(Ld[b] - Lp[0, :, L - 1])) <= 1e-15
    # an empty sequence gives O = 0 and LSE = -inf
    Oz, Lz = oracle.decode(q[:1], Kc[:0], Vc[:0], np.array([0], np.int32), 0.4, lib=lib)
    assert np.all(Oz == 0.0) and np.all(np.isneginf(Lz))


def check_page_causal_count(lib):
    """Page 3, section 1: at S=2048 the causal mask keeps ~2.09M of ~4.19M scores."""
    with open(os.path.join(GOLDEN, "page3_causal_counts.json")) as f:
        g = json.load(f)
    S = g["seq_len"]
    # Q = K = 0 and V = identity: row i of O is the attention row, 1/(i+1) on j <= i
    Q = np.zeros((1, 1, S, S), np.float32)
    V = np.eye(S, dtype=np.float32)[None, None]
    O, _ = oracle.attention(Q, Q, V, 1.0, True, lib=lib)
    kept = int(np.count_nonzero(O))
    assert O.size == g["scores_total"]
    assert abs(kept - g["scores_kept_approx"]) <= g["approx_tolerance"] * g["scores_kept_approx"]
    assert kept == S * (S + 1) // 2


def check_key_lens_bruteforce_decimal(lib):
    """Key padding against the 50-digit brute force, empty sequences included."""
    rng = np.random.default_rng(17)
    for causal in (True, False):
        for (B, H, S, D), kl in (((3, 1, 6, 3), [6, 2, 0]), ((2, 2, 5, 2), [1, 4])):
            Q = rng.standard_normal((B, H, S, D)).astype(np.float32)
            K = rng.standard_normal((B, H, S, D)).astype(np.float32)
            V = rng.standard_normal((B, H, S, D)).astype(np.float32)
            O, L = oracle.attention(Q, K, V, 0.6, causal, lib=lib, key_lens=kl)
            Ob, Lb = _decimal_attention(Q, K, V, 0.6, causal, key_lens=kl)
            assert np.max(np.abs(O - Ob)) <= 1e-13, ("O", causal, kl)
            fin = np.isfinite(Lb)
            assert np.array_equal(np.isfinite(L), fin), ("LSE finite", causal, kl)
            assert np.max(np.abs(L[fin] - Lb[fin])) <= 1e-13, ("LSE", causal, kl)
            assert np.all(L[~fin] == -np.inf)


def check_key_lens_library_softmax(lib):
    """Key padding against scipy's softmax / logsumexp on the masked scores."""
    from scipy.special import logsumexp, softmax
    rng = np.random.default_rng(19)
    B, H, S, D = 3, 2, 41, 8
    kl = np.array([41, 17, 1], np.int32)
    Q = (2 * rng.standard_normal((B, H, S, D))).astype(np.float32)
    K = (2 * rng.standard_normal((B, H, S, D))).astype(np.float32)
    V = rng.standard_normal((B, H, S, D)).astype(np.float32)
    scale = 1 / math.sqrt(D)
    for causal in (True, False):
        O, L = oracle.attention(Q, K, V, scale, causal, lib=lib, key_lens=kl)
        s = scale * np.einsum("bhid,bhjd->bhij", Q.astype(np.float64), K.astype(np.float64))
        keep = np.arange(S)[None, None, None, :] < kl[:, None, None, None]
        if causal:
            keep = keep & np.tril(np.ones((S, S), dtype=bool))[None, None]
        s = np.where(keep, s, -np.inf)
        Oref = softmax(s, axis=-1) @ V.astype(np.float64)
        Lref = logsumexp(s, axis=-1)
        assert np.max(np.abs(O - Oref)) <= 1e-12, causal
        assert np.max(np.abs(L - Lref)) <= 1e-12, causal


def check_key_lens_zero_query_mean(lib):
    """Q = 0: every valid key has the same weight, so O_i is the mean of the
    first n values and LSE_i = ln n, n = min(i + 1, L_b) (causal) or L_b."""
    rng = np.random.default_rng(23)
    B, H, S, D = 3, 2, 13, 4
    kl = np.array([13, 5, 1], np.int32)
    Q = np.zeros((B, H, S, D), np.float32)
    K = rng.standard_normal((B, H, S, D)).astype(np.float32)
    V = rng.standard_normal((B, H, S, D)).astype(np.float32)
    Vd = V.astype(np.float64)
    for causal in (True, False):
        O, L = oracle.attention(Q, K, V, 0.5, causal, lib=lib, key_lens=kl)
        for b in range(B):
            for i in range(S):
                n = min(i + 1, int(kl[b])) if causal else int(kl[b])
                assert np.max(np.abs(O[b, :, i] - Vd[b, :, :n].mean(axis=1))) <= 1e-14
                assert np.max(np.abs(L[b, :, i] - math.log(n))) <= 1e-14


def check_padding_keys_do_not_matter(lib):
    """Keys at or past L_b are padding: replacing their K and V rows by other
    numbers changes nothing, bit for bit."""
    rng = np.random.default_rng(29)
    B, H, S, D = 2, 3, 23, 6
    kl = np.array([9, 23], np.int32)
    Q, K, V = (rng.standard_normal((B, H, S, D)).astype(np.float32) for _ in range(3))
    K2, V2 = K.copy(), V.copy()
    K2[0, :, 9:] = 50 * rng.standard_normal((H, S - 9, D))
    V2[0, :, 9:] = 1e3
    for causal in (True, False):
        O, L = oracle.attention(Q, K, V, 0.4, causal, lib=lib, key_lens=kl)
        O2, L2 = oracle.attention(Q, K2, V2, 0.4, causal, lib=lib, key_lens=kl)
        assert np.array_equal(O, O2) and np.array_equal(L, L2), causal


def check_qkv_bruteforce_fsum(lib):
    """The fused projection against an exactly rounded sum (math.fsum of the
    exact double products of float32 values) on a tiny case."""
    rng = np.random.default_rng(31)
    B, S, hid, H, D = 2, 3, 5, 2, 2
    X = rng.standard_normal((B, S, hid)).astype(np.float32)
    W = rng.standard_normal((hid, 3 * H * D)).astype(np.float32)
    Q, K, V = oracle.qkv_projection(X, W, H, D)
    out = (Q, K, V)
    for b in range(B):
        for s_ in range(S):
            for c in range(3):
                for h in range(H):
                    for d in range(D):
                        n = c * H * D + h * D + d
                        ref = math.fsum(float(X[b, s_, k]) * float(W[k, n]) for k in range(hid))
                        assert abs(out[c][b, h, s_, d] - ref) <= 1e-14 * (1 + abs(ref))


def check_qkv_selection_and_layout(lib):
    """One-hot weights copy chosen input features exactly; one-hot inputs
    reproduce rows of W, placed at [c][b, h, s, d] with n = c*H*D + h*D + d."""
    rng = np.random.default_rng(37)
    B, S, hid, H, D = 2, 4, 6, 3, 2
    N = 3 * H * D
    X = rng.standard_normal((B, S, hid)).astype(np.float32)
    pick = rng.integers(0, hid, size=N)
    W = np.zeros((hid, N), np.float32)
    W[pick, np.arange(N)] = 1.0
    Q, K, V = oracle.qkv_projection(X, W, H, D)
    for c, T in enumerate((Q, K, V)):
        for h in range(H):
            for d in range(D):
                n = c * H * D + h * D + d
                assert np.array_equal(T[:, h, :, d], X[:, :, pick[n]].astype(np.float64))
    W2 = rng.standard_normal((hid, N)).astype(np.float32)
    X2 = np.zeros((B, S, hid), np.float32)
    X2[1, 2, 4] = 1.0
    Q, K, V = oracle.qkv_projection(X2, W2, H, D)
    row = W2[4].astype(np.float64).reshape(3, H, D)
    for c, T in enumerate((Q, K, V)):
        assert np.array_equal(T[1, :, 2, :], row[c])
        mask = np.ones(T.shape, bool)
        mask[1, :, 2, :] = False
        assert np.all(T[mask] == 0.0)


def check_out_proj_bruteforce_fsum(lib):
    """The output projection against exactly rounded sums on a tiny case."""
    rng = np.random.default_rng(41)
    B, H, S, D, N = 2, 3, 4, 2, 5
    O = rng.standard_normal((B, H, S, D)).astype(np.float32)
    W = rng.standard_normal((H * D, N)).astype(np.float32)
    Y = oracle.out_projection(O, W)
    for b in range(B):
        for s_ in range(S):
            for n in range(N):
                ref = math.fsum(float(O[b, h, s_, d]) * float(W[h * D + d, n])
                                for h in range(H) for d in range(D))
                assert abs(Y[b, s_, n] - ref) <= 1e-14 * (1 + abs(ref))


def check_out_proj_head_order(lib):
    """A single 1 at O[b, h, s, d] makes row (b, s) of Y row h*D + d of W_O
    and every other row zero: the heads are concatenated head-major."""
    rng = np.random.default_rng(43)
    B, H, S, D, N = 2, 3, 5, 4, 6
    W = rng.standard_normal((H * D, N)).astype(np.float32)
    for (b, h, s_, d) in ((1, 2, 3, 1), (0, 0, 0, 3), (1, 1, 4, 0)):
        O = np.zeros((B, H, S, D), np.float32)
        O[b, h, s_, d] = 1.0
        Y = oracle.out_projection(O, W)
        assert np.array_equal(Y[b, s_], W[h * D + d].astype(np.float64))
        Y[b, s_] = 0.0
        assert not np.any(Y)


ALL_CHECKS = [
    check_bruteforce_decimal,
    check_library_softmax,
    check_zero_query_prefix_mean,
    check_row0_and_two_keys,
    check_constant_v,
    check_identity_values_give_probabilities,
    check_key_shift_invariance,
    check_joint_permutation,
    check_causal_row_is_prefix_attention,
    check_scale_folding,
    check_rows_subset,
    check_decode_is_last_causal_row,
    check_page_causal_count,
    check_key_lens_bruteforce_decimal,
    check_key_lens_library_softmax,
    check_key_lens_zero_query_mean,
    check_padding_keys_do_not_matter,
    check_qkv_bruteforce_fsum,
    check_qkv_selection_and_layout,
    check_out_proj_bruteforce_fsum,
    check_out_proj_head_order,
]
