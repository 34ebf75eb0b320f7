"""Pins for the CPU oracle: checks against what the pages and plain mathematics fix, not against
the oracle's own code.  Each ``pin_*`` function raises AssertionError when the oracle (the module
passed in) disagrees.  ``tests/test_oracle_pins.py`` runs them on the real oracle and
``tests/test_oracle_mutants.py`` runs them on deliberately broken copies, which must fail.

Sources: SparseSpec ("Accelerating Large-Scale Reasoning Model Inference: Self-Speculative
Decoding with Sparse Attention") §4.1 (verify dumps scores, GQA reduction, Top-K, draft over the
selected tokens) and §4.2 (paged KV; sparse and full attention are one pipeline); SpecSA post,
overlap-aware grouped query execution (candidates share KV blocks); SparDA §2 (max-pool to the
selection grid).
"""

from __future__ import annotations

import math

import numpy as np


# ----------------------------------------------------------------------------------------------
# Input construction (layout only).
# ----------------------------------------------------------------------------------------------

def paged_from_contiguous(Ks, Vs, page_size, shuffle_seed=None, spare=0):
    """Ks, Vs: lists (per request) of [H_kv, L_b, d] float32 arrays.  Returns pool (float32,
    [P, 2, H_kv, page_size, d], NaN in unused slots), page_table [B, max_pages] (-1 unused) and
    seq_lens [B]."""
    B = len(Ks)
    h_kv, _, d = Ks[0].shape
    lens = [k.shape[1] for k in Ks]
    npages = [(L + page_size - 1) // page_size for L in lens]
    total = sum(npages) + spare
    order = (np.random.default_rng(shuffle_seed).permutation(total) if shuffle_seed is not None
             else np.arange(total))
    pool = np.full((total, 2, h_kv, page_size, d), np.nan, np.float32)
    pt = np.full((B, max(1, max(npages))), -1, np.int32)
    off = 0
    for b in range(B):
        for j in range(npages[b]):
            p = int(order[off + j])
            pt[b, j] = p
            for slot in range(page_size):
                t = j * page_size + slot
                if t < lens[b]:
                    pool[p, 0, :, slot, :] = Ks[b][:, t, :]
                    pool[p, 1, :, slot, :] = Vs[b][:, t, :]
        off += npages[b]
    return pool, pt, np.array(lens, np.int32)


def rand_case(rng, B, lens, h_q, h_kv, d, n_c):
    Ks = [rng.standard_normal((h_kv, L, d)).astype(np.float32) for L in lens]
    Vs = [rng.standard_normal((h_kv, L, d)).astype(np.float32) for L in lens]
    q = rng.standard_normal((B, n_c, h_q, d)).astype(np.float32)
    return Ks, Vs, q


# ----------------------------------------------------------------------------------------------
# Independent formulations used as comparators.
# ----------------------------------------------------------------------------------------------

def brute_verify(Ks, Vs, q, scale):
    """Explicit masked score matrix per query head on contiguous KV: S[i, t] = scale q_i . k_t,
    -inf where t > L - n_c + i, row softmax, out = P V, crit[g] = column sums of P over the heads
    that read KV head g."""
    B, n_c, h_q, d = q.shape
    h_kv = Ks[0].shape[0]
    G = h_q // h_kv
    Lmax = max(k.shape[1] for k in Ks)
    out = np.zeros((B, n_c, h_q, d))
    crit = np.zeros((B, h_kv, Lmax))
    crit_cand = np.zeros((B, h_kv, n_c, Lmax))
    for b in range(B):
        L = Ks[b].shape[1]
        tt = np.arange(L)[None, :]
        ii = np.arange(n_c)[:, None]
        mask = tt > (L - n_c + ii)
        for h in range(h_q):
            g = h // G
            K = Ks[b][g].astype(np.float64)
            V = Vs[b][g].astype(np.float64)
            S = scale * (q[b, :, h, :].astype(np.float64) @ K.T)
            S[mask] = -np.inf
            P = np.exp(S - S.max(axis=1, keepdims=True))
            P /= P.sum(axis=1, keepdims=True)
            out[b, :, h, :] = P @ V
            crit[b, g, :L] += P.sum(axis=0)
            crit_cand[b, g, :, :L] += P
    return out, crit, crit_cand


# ----------------------------------------------------------------------------------------------
# Pins.
# ----------------------------------------------------------------------------------------------

def pin_softmax_closed_form(orc):
    """Three tokens with logits 0, 1, 2 (q = [1, 0], k_t = [t, 0], scale 1): p = e^t / (1+e+e^2),
    out = sum_t p_t v_t and lse = log(1 + e + e^2)."""
    K = np.array([[[0, 0], [1, 0], [2, 0]]], np.float32)
    V = np.array([[[1, 0], [0, 1], [0, 0]]], np.float32)
    q = np.array([[[[1, 0]]]], np.float32)  # B=1, n_c=1, H_q=1, d=2
    pool, pt, sl = paged_from_contiguous([K], [V], 2)
    r = orc.verify(orc.PagedKV(pool, pt, sl), q, 1.0)
    z = 1 + math.e + math.e ** 2
    p = [1 / z, math.e / z, math.e ** 2 / z]
    np.testing.assert_allclose(r["out"][0, 0, 0], [p[0], p[1]], rtol=0, atol=1e-14)
    np.testing.assert_allclose(r["crit"][0, 0, :3], p, rtol=0, atol=1e-14)
    assert abs(r["lse"][0, 0, 0] - math.log(z)) < 1e-14


def pin_brute_force(orc):
    """Tiny random cases (B=2, L<=12, d=4, G in {1,2}, n_c in {1,2,3}) against brute_verify."""
    rng = np.random.default_rng(7)
    for G in (1, 2):
        for n_c in (1, 2, 3):
            lens = [int(rng.integers(n_c, 13)), int(rng.integers(n_c, 13))]
            Ks, Vs, q = rand_case(rng, 2, lens, 2 * G, 2, 4, n_c)
            pool, pt, sl = paged_from_contiguous(Ks, Vs, 4, shuffle_seed=3)
            r = orc.verify(orc.PagedKV(pool, pt, sl), q, 0.5, per_candidate=True)
            out, crit, cc = brute_verify(Ks, Vs, q, 0.5)
            np.testing.assert_allclose(r["out"], out, rtol=0, atol=1e-12)
            np.testing.assert_allclose(r["crit"], crit, rtol=0, atol=1e-12)
            np.testing.assert_allclose(r["crit_cand"], cc, rtol=0, atol=1e-12)


def pin_identical_keys(orc):
    """All keys equal: every visible token gets probability 1/|vis_i|, so out_i is the mean of the
    visible V rows, lse_i = s + log|vis_i|, and crit_t = sum over i with t visible of G/|vis_i|."""
    rng = np.random.default_rng(11)
    B, h_q, h_kv, d, n_c = 2, 4, 2, 8, 3
    G = h_q // h_kv
    lens = [9, 6]
    kvec = rng.standard_normal(d).astype(np.float32)
    Ks = [np.broadcast_to(kvec, (h_kv, L, d)).copy() for L in lens]
    Vs = [rng.standard_normal((h_kv, L, d)).astype(np.float32) for L in lens]
    q = rng.standard_normal((B, n_c, h_q, d)).astype(np.float32)
    pool, pt, sl = paged_from_contiguous(Ks, Vs, 4, shuffle_seed=5)
    scale = 0.3
    r = orc.verify(orc.PagedKV(pool, pt, sl), q, scale)
    for b, L in enumerate(lens):
        for i in range(n_c):
            nvis = L - n_c + i + 1
            for h in range(h_q):
                g = h // G
                np.testing.assert_allclose(r["out"][b, i, h], Vs[b][g, :nvis].astype(np.float64).mean(0),
                                           rtol=0, atol=1e-12)
                s = scale * float(np.dot(q[b, i, h].astype(np.float64), kvec.astype(np.float64)))
                assert abs(r["lse"][b, i, h] - (s + math.log(nvis))) < 1e-12
        for g in range(h_kv):
            want = np.zeros(L)
            for i in range(n_c):
                nvis = L - n_c + i + 1
                want[:nvis] += G / nvis
            np.testing.assert_allclose(r["crit"][b, g, :L], want, rtol=0, atol=1e-12)


def pin_crit_sums(orc):
    """sum_t crit[b,g,t] = n_c * G and sum_t crit_cand[b,g,i,t] = G for every unit."""
    rng = np.random.default_rng(13)
    lens = [17, 33, 5]
    Ks, Vs, q = rand_case(rng, 3, lens, 6, 2, 8, 5)
    pool, pt, sl = paged_from_contiguous(Ks, Vs, 8, shuffle_seed=1)
    r = orc.verify(orc.PagedKV(pool, pt, sl), q, 0.35, per_candidate=True)
    np.testing.assert_allclose(r["crit"].sum(-1), np.full((3, 2), 5 * 3.0), rtol=0, atol=1e-9)
    np.testing.assert_allclose(r["crit_cand"].sum(-1), np.full((3, 2, 5), 3.0), rtol=0, atol=1e-9)


def pin_causality(orc):
    """Changing K/V at positions after L - n_c + i, or the query of any other candidate, leaves
    candidate i's output bit-identical."""
    rng = np.random.default_rng(17)
    lens = [10]
    n_c = 4
    Ks, Vs, q = rand_case(rng, 1, lens, 2, 1, 4, n_c)
    pool, pt, sl = paged_from_contiguous(Ks, Vs, 4)
    base = orc.verify(orc.PagedKV(pool, pt, sl), q, 0.5)
    L = lens[0]
    for i in range(n_c):
        K2 = Ks[0].copy()
        V2 = Vs[0].copy()
        K2[:, L - n_c + i + 1:] += 3.0
        V2[:, L - n_c + i + 1:] -= 2.0
        q2 = q.copy()
        q2[:, [j for j in range(n_c) if j != i]] *= -1.5
        pool2, pt2, sl2 = paged_from_contiguous([K2], [V2], 4)
        r = orc.verify(orc.PagedKV(pool2, pt2, sl2), q2, 0.5)
        assert np.array_equal(r["out"][:, i], base["out"][:, i]), f"candidate {i} saw a later position"
        assert np.array_equal(r["lse"][:, i], base["lse"][:, i])


def pin_paging_invariance(orc):
    """A shuffled page table with spare pages gives exactly the identity-table result."""
    rng = np.random.default_rng(19)
    lens = [23, 40]
    Ks, Vs, q = rand_case(rng, 2, lens, 4, 2, 8, 2)
    a = orc.verify(orc.PagedKV(*paged_from_contiguous(Ks, Vs, 8)), q, 0.4)
    b = orc.verify(orc.PagedKV(*paged_from_contiguous(Ks, Vs, 8, shuffle_seed=4, spare=3)), q, 0.4)
    for key in ("out", "lse", "crit"):
        assert np.array_equal(a[key], b[key])


def pin_gqa_equals_mha(orc):
    """GQA with group G equals MHA on a cache whose head h is a copy of KV head h // G; the GQA
    criticality of group g is the sum of the MHA criticality of its G heads."""
    rng = np.random.default_rng(23)
    G, h_kv, d, n_c = 3, 2, 4, 2
    lens = [11, 7]
    Ks, Vs, q = rand_case(rng, 2, lens, G * h_kv, h_kv, d, n_c)
    gqa = orc.verify(orc.PagedKV(*paged_from_contiguous(Ks, Vs, 4, shuffle_seed=2)), q, 0.6)
    Km = [np.repeat(k, G, axis=0) for k in Ks]
    Vm = [np.repeat(v, G, axis=0) for v in Vs]
    mha = orc.verify(orc.PagedKV(*paged_from_contiguous(Km, Vm, 4)), q, 0.6)
    np.testing.assert_allclose(gqa["out"], mha["out"], rtol=0, atol=1e-13)
    summed = mha["crit"].reshape(2, h_kv, G, -1).sum(2)
    np.testing.assert_allclose(gqa["crit"], summed, rtol=0, atol=1e-13)


def pin_draft_select_all(orc):
    """A draft over every index 0..L-1 is single-query dense attention: it equals verify with
    n_c = 1 on the same query, and brute force."""
    rng = np.random.default_rng(29)
    lens = [13, 6]
    Ks, Vs, q = rand_case(rng, 2, lens, 4, 2, 8, 1)
    kv = orc.PagedKV(*paged_from_contiguous(Ks, Vs, 4, shuffle_seed=8))
    k_max = 16
    idx = np.full((2, 2, k_max), -1, np.int32)
    cnt = np.zeros((2, 2), np.int32)
    for b, L in enumerate(lens):
        idx[b, :, :L] = np.arange(L)
        cnt[b, :] = L
    dr = orc.draft(kv, q[:, 0], idx, cnt, 0.45)
    vr = orc.verify(kv, q, 0.45)
    bf, _, _ = brute_verify(Ks, Vs, q, 0.45)
    np.testing.assert_allclose(dr["out"], vr["out"][:, 0], rtol=0, atol=1e-13)
    np.testing.assert_allclose(dr["out"], bf[:, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dr["lse"], vr["lse"][:, 0], rtol=0, atol=1e-13)


def pin_draft_subset(orc):
    """A draft over an index subset equals brute-force softmax attention restricted to it."""
    rng = np.random.default_rng(31)
    lens = [20]
    Ks, Vs, q = rand_case(rng, 1, lens, 2, 1, 4, 1)
    kv = orc.PagedKV(*paged_from_contiguous(Ks, Vs, 8, shuffle_seed=9))
    sub = np.array([0, 3, 4, 11, 19], np.int32)
    idx = np.full((1, 1, 8), -1, np.int32)
    idx[0, 0, :5] = sub
    cnt = np.array([[5]], np.int32)
    dr = orc.draft(kv, q[:, 0], idx, cnt, 0.7)
    for h in range(2):
        K = Ks[0][0, sub].astype(np.float64)
        V = Vs[0][0, sub].astype(np.float64)
        s = 0.7 * (K @ q[0, 0, h].astype(np.float64))
        p = np.exp(s - s.max())
        p /= p.sum()
        np.testing.assert_allclose(dr["out"][0, h], p @ V, rtol=0, atol=1e-13)


def pin_draft_duplicates(orc):
    """An index listed twice counts twice (the ABI's stated convention): the draft equals softmax
    attention in which that token's weight is doubled, i.e. its logit raised by ln 2, and the
    log-sum-exp includes both copies."""
    rng = np.random.default_rng(37)
    Ks, Vs, q = rand_case(rng, 1, [9], 2, 1, 4, 1)
    kv = orc.PagedKV(*paged_from_contiguous(Ks, Vs, 4, shuffle_seed=3))
    idx = np.full((1, 1, 4), -1, np.int32)
    idx[0, 0, :3] = [2, 2, 7]
    cnt = np.array([[3]], np.int32)
    dr = orc.draft(kv, q[:, 0], idx, cnt, 0.6)
    K = Ks[0][0, [2, 7]].astype(np.float64)
    V = Vs[0][0, [2, 7]].astype(np.float64)
    for h in range(2):
        s = 0.6 * (K @ q[0, 0, h].astype(np.float64)) + np.array([math.log(2.0), 0.0])
        m = s.max()
        w = np.exp(s - m)
        np.testing.assert_allclose(dr["out"][0, h], (w / w.sum()) @ V, rtol=0, atol=1e-13)
        np.testing.assert_allclose(dr["lse"][0, h], m + math.log(w.sum()), rtol=0, atol=1e-12)


def pin_topk(orc):
    """Top-K special cases and a brute-force comparison with Python's sort."""
    rng = np.random.default_rng(37)
    # K = L keeps everything; constant scores keep 0..K-1; K = 1 is the first argmax.
    s = rng.random((1, 9)).astype(np.float32)
    idx, cnt = orc.topk(s, [9], [9], 9)
    assert cnt[0] == 9 and list(idx[0]) == list(range(9))
    c = np.full((1, 12), 0.25, np.float32)
    idx, cnt = orc.topk(c, [12], [5], 6)
    assert list(idx[0]) == [0, 1, 2, 3, 4, -1] and cnt[0] == 5
    a = np.array([[0.1, 0.9, 0.3, 0.9, 0.2]], np.float32)
    idx, _ = orc.topk(a, [5], [1], 1)
    assert idx[0, 0] == 1
    idx, _ = orc.topk(a, [5], [3], 3)
    assert list(idx[0]) == [1, 2, 3]
    # Brute force on rows with many ties; a row may be shorter than the stride (lens per group).
    for trial in range(30):
        n = int(rng.integers(1, 40))
        k = int(rng.integers(0, n + 1))
        row = rng.integers(0, 4, size=(1, 48)).astype(np.float32) / 4
        idx, cnt = orc.topk(row, [n], [k], 48)
        order = sorted(range(n), key=lambda t: (-float(row[0, t]), t))[:k]
        assert cnt[0] == k
        assert list(idx[0, :k]) == sorted(order)
        assert all(v == -1 for v in idx[0, k:])


def pin_block_maxpool(orc):
    """Block size 1 reproduces the per-candidate criticality; larger blocks take the maximum over
    each block, the last block possibly partial."""
    rng = np.random.default_rng(41)
    lens = [19]
    Ks, Vs, q = rand_case(rng, 1, lens, 4, 2, 4, 3)
    kv = orc.PagedKV(*paged_from_contiguous(Ks, Vs, 4, shuffle_seed=3))
    r = orc.verify(kv, q, 0.5, per_candidate=True)
    cc = r["crit_cand"]
    b1 = orc.block_maxpool(cc, kv.seq_lens, 1)
    np.testing.assert_array_equal(b1[..., :19], cc[..., :19])
    b8 = orc.block_maxpool(cc, kv.seq_lens, 8)
    assert b8.shape[-1] == 3
    for j in range(3):
        np.testing.assert_array_equal(b8[..., j], cc[..., 8 * j:min(8 * j + 8, 19)].max(-1))


def pin_block_union(orc):
    """The union is the sorted set of all candidates' blocks; the mask bit i marks candidate i's
    blocks; identical sets give that set with every bit set."""
    blocks = np.array([[[5, 1, 9], [1, 2, 9], [7, 5, 0]]], np.int32)  # U=1, n_c=3, kb=3
    bcnt = np.array([[3, 3, 2]], np.int32)
    uidx, umask, ucnt = orc.block_union(blocks, bcnt)
    assert ucnt[0] == 5
    assert list(uidx[0, :5]) == [1, 2, 5, 7, 9]
    assert list(umask[0, :5]) == [0b011, 0b010, 0b101, 0b100, 0b011]
    same = np.array([[[4, 2], [4, 2]]], np.int32)
    uidx, umask, ucnt = orc.block_union(same, np.array([[2, 2]], np.int32))
    assert ucnt[0] == 2 and list(uidx[0, :2]) == [2, 4] and list(umask[0, :2]) == [3, 3]


def pin_block_attn(orc):
    """With every block selected, block-sparse attention is the verify attention; with a subset it
    is brute-force softmax over that candidate's own visible tokens."""
    rng = np.random.default_rng(43)
    lens = [21]
    n_c, bs = 3, 4
    Ks, Vs, q = rand_case(rng, 1, lens, 4, 2, 4, n_c)
    kv = orc.PagedKV(*paged_from_contiguous(Ks, Vs, 4, shuffle_seed=6))
    nb = 6
    allb = np.tile(np.arange(nb, dtype=np.int32), (1, 2, n_c, 1))
    ball = orc.block_attn(kv, q, allb, np.full((1, 2, n_c), nb, np.int32), bs, 0.5)
    vr = orc.verify(kv, q, 0.5)
    np.testing.assert_allclose(ball["out"], vr["out"], rtol=0, atol=1e-13)
    sel = np.array([[[[0, 5], [2, 3], [5, 1]]] * 2], np.int32).reshape(1, 2, n_c, 2)
    bsub = orc.block_attn(kv, q, sel, np.full((1, 2, n_c), 2, np.int32), bs, 0.5)
    L = lens[0]
    for h in range(4):
        g = h // 2
        for i in range(n_c):
            toks = [t for t in range(L) if t // bs in set(sel[0, g, i]) and t <= L - n_c + i]
            K = Ks[0][g, toks].astype(np.float64)
            V = Vs[0][g, toks].astype(np.float64)
            s = 0.5 * (K @ q[0, i, h].astype(np.float64))
            p = np.exp(s - s.max())
            p /= p.sum()
            np.testing.assert_allclose(bsub["out"][0, i, h], p @ V, rtol=0, atol=1e-13)


def _kv_case(rng, lens, n, h_kv=2, d=8, ps=4, shuffle_seed=3):
    """Full sequences of L + n tokens, their paged cache, and the 'before' cache in which the last n
    slots of every request are blank (NaN): appending those n tokens must reproduce the full cache."""
    Ks = [rng.standard_normal((h_kv, L + n, d)).astype(np.float32) for L in lens]
    Vs = [rng.standard_normal((h_kv, L + n, d)).astype(np.float32) for L in lens]
    full, pt, full_lens = paged_from_contiguous(Ks, Vs, ps, shuffle_seed=shuffle_seed)
    before = full.copy()
    for b, L in enumerate(lens):
        for t in range(L, L + n):
            before[pt[b, t // ps], :, :, t % ps, :] = np.nan
    k_new = np.stack([Ks[b][:, L:L + n, :].transpose(1, 0, 2) for b, L in enumerate(lens)])
    v_new = np.stack([Vs[b][:, L:L + n, :].transpose(1, 0, 2) for b, L in enumerate(lens)])
    return Ks, Vs, full, before, pt, full_lens, k_new, v_new


def pin_kv_append_composes(orc):
    """Appending each request's next n tokens to a paged cache reproduces the cache built directly
    from the longer sequences (every other pool element untouched), and verifying with the appended
    tokens as the candidates equals brute force on the contiguous sequences.  Appending nothing
    changes nothing."""
    rng = np.random.default_rng(53)
    lens, n, G = [5, 9], 3, 2
    Ks, Vs, full, before, pt, full_lens, k_new, v_new = _kv_case(rng, lens, n)
    max_len = pt.shape[1] * 4
    after, ok = orc.kv_append(before, pt, np.array(lens, np.int32), max_len, k_new, v_new)
    assert ok.tolist() == [1, 1]
    np.testing.assert_array_equal(after, full)
    q = rng.standard_normal((2, n, 2 * G, 8)).astype(np.float32)
    res = orc.verify(orc.PagedKV(after, pt, full_lens), q, 0.3)
    ref_out, _, _ = brute_verify(Ks, Vs, q, 0.3)
    assert np.allclose(res["out"], ref_out, rtol=0, atol=1e-12)
    same, ok0 = orc.kv_append(before, pt, np.array(lens, np.int32), max_len, k_new[:, :0], v_new[:, :0])
    assert ok0.tolist() == [1, 1]
    np.testing.assert_array_equal(same, before)


def pin_kv_append_skips(orc):
    """A request whose new tokens would pass max_seq_len, or reach a skipped page, is left
    untouched; the others are written."""
    rng = np.random.default_rng(59)
    lens, n = [10, 4, 2], 3
    _, _, full, before, pt, _, k_new, v_new = _kv_case(rng, lens, n)
    pt = pt.copy()
    pt[2, (lens[2] + 1) // 4] = -1  # request 2: its second new token falls in a missing page
    after, ok = orc.kv_append(before, pt, np.array(lens, np.int32), 12, k_new, v_new)
    assert ok.tolist() == [0, 1, 0]
    for b, L in enumerate(lens):
        for t in range(L, L + n):
            p = pt[b, t // 4]
            if p < 0:
                continue
            want = full if b == 1 else before
            np.testing.assert_array_equal(after[p, :, :, t % 4, :], want[p, :, :, t % 4, :])


def pin_kv_advance(orc):
    """Advancing by +n then -n is the identity; a result outside [0, max_seq_len] leaves the
    length unchanged; accepting a of n_c candidates is an advance by -(n_c - a)."""
    lens = np.array([5, 9, 0, 12], np.int32)
    up = orc.kv_advance(lens, np.array([3, 3, 3, 1], np.int32), 12)
    assert up.tolist() == [8, 12, 3, 12]
    back = orc.kv_advance(up, np.array([-3, -3, -3, 0], np.int32), 12)
    assert back.tolist() == [5, 9, 0, 12]
    assert orc.kv_advance(lens, np.array([-6, 0, -1, 0], np.int32), 12).tolist() == [5, 9, 0, 12]
    n_c, accepted = 5, np.array([2, 5, 0, 1], np.int32)
    cand = orc.kv_advance(np.array([10, 10, 10, 10], np.int32), np.full(4, n_c, np.int32), 64)
    assert orc.kv_advance(cand, -(n_c - accepted), 64).tolist() == (10 + accepted).tolist()


def pin_phase_assignment(orc):
    """Arrivals into empty buckets fill them round-robin (offsets 0, 1, ..., k, 0, ...), so the counts
    never differ by more than one; an arrival joins the emptiest bucket, ties to the lowest offset;
    over any n_buckets consecutive steps every request verifies exactly once, and at each step the
    verifying requests are those of one bucket."""
    nb = 5
    c, off = orc.phase_assign(np.zeros(nb, np.int32), 12)
    assert off.tolist() == [0, 1, 2, 3, 4, 0, 1, 2, 3, 4, 0, 1]
    assert c.tolist() == [3, 3, 2, 2, 2] and c.max() - c.min() <= 1
    c2, off2 = orc.phase_assign(np.array([4, 1, 3, 1, 2], np.int32), 3)
    assert off2.tolist() == [1, 3, 1] and c2.tolist() == [4, 3, 3, 2, 2]
    # A request that joins at offset 0 drafts for k = nb - 1 steps, then verifies (a speculative
    # round is k drafts followed by one verify).
    assert [int(orc.phase_flags(np.array([0], np.int32), nb, s)[0]) for s in range(2 * nb)] == [0, 0, 0, 0, 1] * 2
    offsets = np.array([0, 1, 2, 3, 4, 0, 1, 2], np.int32)
    total = np.zeros(len(offsets), np.int64)
    for step in range(3, 3 + nb):
        f = orc.phase_flags(offsets, nb, step)
        total += f
        assert len(set(offsets[f == 1].tolist())) == 1
    assert total.tolist() == [1] * len(offsets)


def pin_topp(orc):
    """Top-p against a brute-force prefix search on sorted rows; p = 1 keeps exactly the non-zero
    entries; equal entries keep ceil(p n) of them, the lowest indices; K never decreases with p;
    K is capped at k_max; a zero row keeps nothing."""
    rng = np.random.default_rng(73)
    s = rng.random((6, 40)).astype(np.float32) ** 3
    s[1, 20:] = 0.0
    s[2, :] = 0.25
    s[3, :] = 0.0
    lens = np.array([40, 40, 40, 40, 17, 1], np.int32)
    for p in (0.0, 0.1, 0.5, 0.9, 0.999, 1.0):
        idx, cnt, k = orc.topp(s, lens, p, 40)
        for r in range(6):
            n = lens[r]
            order = sorted(range(n), key=lambda t: (-float(s[r, t]), t))
            vals = [float(s[r, t]) for t in order]
            target, acc, kk = p * sum(vals), 0.0, 0
            while kk < n and acc < target:
                acc += vals[kk]
                kk += 1
            assert k[r] == kk and cnt[r] == kk
            assert sorted(idx[r, :kk].tolist()) == sorted(order[:kk]) and idx[r, :kk].tolist() == sorted(order[:kk])
    _, _, k1 = orc.topp(s, lens, 1.0, 40)
    assert k1[1] == 20 and k1[3] == 0
    _, _, kq = orc.topp(s, lens, 0.3, 40)
    assert kq[2] == 12  # 0.3 * 40 equal entries
    ks = [orc.topp(s, lens, p, 40)[2] for p in (0.2, 0.4, 0.6, 0.8)]
    assert all((a <= b).all() for a, b in zip(ks, ks[1:]))
    _, capped, kc = orc.topp(s, lens, 1.0, 5)
    assert kc.max() <= 5 and capped.max() <= 5


def pin_combine(orc):
    """Split-KV combine: merging one split is the identity; two splits with equal LSEs average
    their outputs and add ln 2 to the LSE; drafts over disjoint index subsets, merged, equal the
    draft over their union (an empty subset, LSE -inf, changes nothing); a row of only empty
    splits, or of none, gives 0 and -inf."""
    rng = np.random.default_rng(83)
    o1 = rng.standard_normal((3, 1, 8)).astype(np.float32)
    l1 = np.array([[0.25], [-3.5], [-np.inf]], np.float32)
    out, lse = orc.combine(o1, l1)
    np.testing.assert_array_equal(out[:2], o1[:2, 0].astype(np.float64))
    np.testing.assert_array_equal(lse[:2], l1[:2, 0].astype(np.float64))
    assert lse[2] == -np.inf and not out[2].any()
    o2 = rng.standard_normal((1, 2, 8)).astype(np.float32)
    out, lse = orc.combine(o2, np.array([[1.5, 1.5]], np.float32))
    np.testing.assert_allclose(out[0], o2[0].astype(np.float64).mean(axis=0), rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse[0], 1.5 + math.log(2.0), rtol=0, atol=1e-15)
    out, lse = orc.combine(np.zeros((2, 0, 8), np.float32), np.zeros((2, 0), np.float32))
    assert (lse == -np.inf).all() and not out.any()

    Ks, Vs, q = rand_case(rng, 1, [40], 4, 2, 8, 1)
    kv = orc.PagedKV(*paged_from_contiguous(Ks, Vs, 4, shuffle_seed=5))
    sel = np.sort(rng.choice(40, 23, replace=False)).astype(np.int32)
    parts = [sel[:7], sel[7:8], np.zeros(0, np.int32), sel[8:]]
    k_max = 32

    def draft_of(tokens):
        idx = np.full((1, 2, k_max), -1, np.int32)
        idx[0, :, :len(tokens)] = tokens
        cnt = np.full((1, 2), len(tokens), np.int32)
        return orc.draft(kv, q[:, 0], idx, cnt, 0.5)

    ds = [draft_of(t) for t in parts]
    whole = draft_of(sel)
    o_parts = np.stack([d["out"][0] for d in ds], axis=1).astype(np.float32)   # [H_q, S, d]
    l_parts = np.stack([d["lse"][0] for d in ds], axis=1).astype(np.float32)   # [H_q, S]
    assert np.isneginf(l_parts[:, 2]).all()
    out, lse = orc.combine(o_parts, l_parts)
    np.testing.assert_allclose(out, whole["out"][0], rtol=0, atol=2e-6)
    np.testing.assert_allclose(lse, whole["lse"][0], rtol=0, atol=2e-6)


ALL_PINS = [pin_softmax_closed_form, pin_brute_force, pin_identical_keys, pin_crit_sums, pin_causality,
            pin_paging_invariance, pin_gqa_equals_mha, pin_draft_select_all, pin_draft_subset, pin_draft_duplicates,
            pin_topk,
            pin_block_maxpool, pin_block_union, pin_block_attn, pin_kv_append_composes, pin_kv_append_skips,
            pin_kv_advance, pin_phase_assignment, pin_topp, pin_combine]
