"""Pins of the fp64 oracle against facts fixed outside it.

Each ``pin_*`` function raises AssertionError when the oracle (or a
deliberately broken build of it, ``mutant`` > 0) disagrees with something the
mathematics fixes on its own: brute force on tiny inputs, closed forms,
invariants, and a library routine on a special case.  The test module runs
them against the real oracle, and against every planted-mistake build to show
that each mistake is caught by at least one pin.
"""
import json
import math
import os

import numpy as np
import scipy.special
import torch

import oracle
from mla_speculative_decoding_verify_gb300 import inputs as I

from brute import ancestor_matrix, brute, logical_kv

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _tiny(seed, B=2, H=2, page_size=2, tree_kind="forest", max_p=5, max_t=6, **kw):
    rng = np.random.default_rng(seed)
    prefix = rng.integers(0, max_p + 1, size=B).tolist()
    trees = rng.integers(1, max_t + 1, size=B).tolist()
    return I.make_inputs(prefix, trees, tree_kind=tree_kind, page_size=page_size, seed=seed,
                         stream=7, num_heads=H, **kw)


def pin_brute(mutant=0):
    """Oracle == independent brute force (closure mask, unshifted fsum softmax)."""
    for seed in range(4):
        for kind in ("forest", "uniform", "chain"):
            inp = _tiny(seed, tree_kind=kind)
            o, l = oracle.verify(inp, mutant=mutant)
            bo, bl = brute(inp)
            np.testing.assert_allclose(l, bl, rtol=0, atol=1e-11)
            np.testing.assert_allclose(o, bo, rtol=0, atol=1e-11)


def pin_single_key(mutant=0):
    """P = 0 and a one-node tree: the only visible key is the node's own, so
    out is exactly its c_kv and lse is its scaled score."""
    inp = I.make_inputs([0, 0, 0], [1, 1, 1], tree_kind="roots", page_size=2, seed=3,
                        stream=8, num_heads=3)
    o, l = oracle.verify(inp, mutant=mutant)
    ql = I.bf16_bits_to_f64(inp.q_lat)
    qr = I.bf16_bits_to_f64(inp.q_rope)
    for b in range(3):
        kv = logical_kv(inp, b)
        for h in range(3):
            q = np.concatenate([ql[b, h], qr[b, h]])
            s = inp.scale * math.fsum(q * kv[0])
            assert np.array_equal(o[b, h], kv[0, :512]), "single key must return its V"
            assert abs(l[b, h] - s) <= 1e-12 * max(1.0, abs(s))


def pin_uniform(mutant=0):
    """q = 0 makes every score 0: out is the plain mean of the visible c_kv rows
    and lse = ln |visible|.  Roots see prefix + self; chain node i sees P + i + 1 keys."""
    for kind in ("roots", "chain"):
        inp = I.make_inputs([5, 0, 3], [4, 3, 5], tree_kind=kind, page_size=2, seed=5,
                            stream=9, num_heads=2, q_zero=True)
        o, l = oracle.verify(inp, mutant=mutant)
        off = 0
        for b in range(inp.batch):
            T = int(inp.n_tree[b])
            P = int(inp.seq_lens[b]) - T
            kv = logical_kv(inp, b)
            for i in range(T):
                vis = list(range(P)) + ([P + i] if kind == "roots" else
                                        list(range(P, P + i + 1)))
                mean = kv[vis, :512].mean(axis=0)
                for h in range(2):
                    np.testing.assert_allclose(o[off + i, h], mean, rtol=0, atol=1e-13)
                    assert abs(l[off + i, h] - math.log(len(vis))) < 1e-13
            off += T


def pin_chain_causal(mutant=0):
    """A chain-shaped tree (parent[i] = i-1) is plain causal masking: node i sees
    keys 0 .. P+i.  The causal reference is scipy's logsumexp over numpy scores."""
    inp = I.make_inputs([37, 12], [9, 5], tree_kind="chain", page_size=8, seed=11, stream=10,
                        num_heads=4)
    o, l = oracle.verify(inp, mutant=mutant)
    ql = I.bf16_bits_to_f64(inp.q_lat)
    qr = I.bf16_bits_to_f64(inp.q_rope)
    off = 0
    for b in range(inp.batch):
        T = int(inp.n_tree[b])
        P = int(inp.seq_lens[b]) - T
        kv = logical_kv(inp, b)
        for i in range(T):
            K = kv[:P + i + 1]
            for h in range(4):
                q = np.concatenate([ql[off + i, h], qr[off + i, h]])
                s = inp.scale * (K @ q)
                ref_l = scipy.special.logsumexp(s)
                ref_o = np.exp(s - ref_l) @ K[:, :512]
                assert abs(l[off + i, h] - ref_l) < 1e-11
                np.testing.assert_allclose(o[off + i, h], ref_o, rtol=0, atol=1e-11)
        off += T


def pin_split(mutant=0):
    """Split-KV partials merged by their log-sum-exp equal the unsplit result
    (random bounds, an empty split, a bound inside the tree keys)."""
    inp = I.make_inputs([23, 9], [7, 6], tree_kind="uniform", page_size=4, seed=13, stream=11,
                        num_heads=2)
    full_o, full_l = oracle.verify_rows(inp, mutant=mutant)
    for bounds in ([0, 5, 5, 17, 26, 31], [0, 1 << 40], [0, 10, 12, 14, 16, 20, 24, 28, 40]):
        po, pl = oracle.split_partials(inp, bounds, mutant=mutant)
        co, cl = oracle.combine(po, pl, mutant=mutant)
        np.testing.assert_allclose(cl, full_l, rtol=0, atol=1e-12)
        np.testing.assert_allclose(co, full_o, rtol=0, atol=1e-12)


def pin_combine_closed_form(mutant=0):
    """Two partials with lse a and b merge to log(e^a + e^b) with logistic weights;
    a partial with lse = -inf has weight 0; all -inf gives 0 and -inf."""
    rng = np.random.default_rng(0)
    po = rng.standard_normal((3, 4, 6))
    pl = np.array([[0.3, -1.0, 2.0, -np.inf],
                   [1.1, -np.inf, 2.0, -np.inf],
                   [-np.inf, -np.inf, -np.inf, -np.inf]])
    o, l = oracle.combine(po, pl, mutant=mutant)
    for r, (a, b) in enumerate([(0.3, 1.1), (-1.0, None), (2.0, 2.0)]):
        if b is None:
            assert l[r] == a
            np.testing.assert_allclose(o[r], po[0, r], rtol=0, atol=1e-15)
            continue
        ref = math.log(math.exp(a) + math.exp(b))
        wa = 1.0 / (1.0 + math.exp(b - a))
        assert abs(l[r] - ref) < 1e-14
        np.testing.assert_allclose(o[r], wa * po[0, r] + (1 - wa) * po[1, r], rtol=0, atol=1e-14)
    assert l[3] == -np.inf and not o[3].any()


def pin_permutation(mutant=0):
    """Re-ordering the prefix tokens leaves every output unchanged (the prefix is a
    set under the mask), and moving pages in the pool changes nothing at all."""
    inp = I.make_inputs([21, 14], [5, 4], tree_kind="forest", page_size=4, seed=17, stream=12,
                        num_heads=2)
    o, l = oracle.verify(inp, mutant=mutant)
    rng = np.random.default_rng(1)
    # 1) physical page permutation with the same logical content
    perm = rng.permutation(inp.num_pages)
    inv = np.argsort(perm)
    moved = I.VerifyInputs(**{**inp.__dict__})
    moved.kv_cache = inp.kv_cache[perm]
    bt = inp.block_table.copy()
    bt[bt >= 0] = inv[bt[bt >= 0]]
    moved.block_table = bt
    o2, l2 = oracle.verify(moved, mutant=mutant)
    assert np.array_equal(o, o2) and np.array_equal(l, l2)
    # 2) logical permutation of each request's prefix rows
    shuffled = I.VerifyInputs(**{**inp.__dict__})
    kv = inp.kv_cache.copy()
    for b in range(inp.batch):
        P = int(inp.seq_lens[b] - inp.n_tree[b])
        if P < 2:
            continue
        slots = [(int(inp.block_table[b, t // 4]), t % 4) for t in range(P)]
        src = [inp.kv_cache[p, r].copy() for p, r in slots]
        order = rng.permutation(P)
        for t, (p, r) in enumerate(slots):
            kv[p, r] = src[order[t]]
    shuffled.kv_cache = kv
    o3, l3 = oracle.verify(shuffled, mutant=mutant)
    np.testing.assert_allclose(l3, l, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o3, o, rtol=0, atol=1e-12)


def pin_torch_library(mutant=0):
    """On a reduced workload-shaped input the oracle equals torch's fp64
    softmax(scale * Q K^T + mask) V with the mask from a boolean matrix power."""
    inp = I.scaled_config_inputs(2, seed=0, prefix_div=64, batch_cap=2)
    o, l = oracle.verify(inp, mutant=mutant)
    ql = torch.from_numpy(I.bf16_bits_to_f64(inp.q_lat))
    qr = torch.from_numpy(I.bf16_bits_to_f64(inp.q_rope))
    off = 0
    for b in range(inp.batch):
        T = int(inp.n_tree[b])
        L = int(inp.seq_lens[b])
        P = L - T
        kv = torch.from_numpy(logical_kv(inp, b))
        par = inp.tree_parent[off:off + T]
        adj = torch.eye(T, dtype=torch.float64)
        for i, p in enumerate(par):
            if p >= 0:
                adj[i, p] = 1.0
        reach = torch.linalg.matrix_power(adj, T) > 0     # ancestor-or-self
        mask = torch.zeros(T, L, dtype=torch.float64)
        mask[:, P:] = torch.where(reach, 0.0, float("-inf"))
        q = torch.cat([ql[off:off + T], qr[off:off + T]], dim=-1)        # [T, H, 576]
        s = inp.scale * torch.einsum("thd,kd->thk", q, kv) + mask[:, None, :]
        ref_l = torch.logsumexp(s, dim=-1)
        ref_o = torch.softmax(s, dim=-1) @ kv[:, :512]
        np.testing.assert_allclose(l[off:off + T], ref_l.numpy(), rtol=0, atol=1e-10)
        np.testing.assert_allclose(o[off:off + T], ref_o.numpy(), rtol=0, atol=1e-10)
        off += T


def _hand_expect(name, scale):
    """Closed forms of tests/golden/hand_worked.json, case by case."""
    ln2, ln3 = math.log(2.0), math.log(3.0)
    if name == "equal_scores_average":
        return [(scale + ln3, {0: 1.0, 1: 2.0})]
    if name == "logistic_pair_rope":
        w = 1.0 / (1.0 + math.exp(-4.0 * scale))
        return [(2.0 * scale + math.log1p(math.exp(-4.0 * scale)), {5: 4.0 * w - 1.0})]
    if name == "sibling_masked":
        return [(0.0, {7: 1.0}), (ln2, {7: 50.5}), (ln2, {7: 0.0})]
    if name == "chain_after_prefix":
        return [(math.log(2.0), {3: 6.0}), (ln3, {3: 14.0 / 3.0}), (math.log(4.0), {3: 3.75})]
    raise KeyError(name)


def pin_golden_hand(mutant=0):
    """Hand-worked cases of tests/golden/hand_worked.json against their closed forms."""
    with open(os.path.join(GOLDEN, "hand_worked.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        H, dl, dr = 1, 512, 64
        P, T = c["prefix"], len(c["parent"])
        L = P + T
        kv = np.zeros((1, L, dl + dr))
        for t, row in c["kv_rows"].items():
            for d, v in row.items():
                kv[0, int(t), int(d)] = v
        q = np.zeros((T, H, dl + dr))
        for i, row in c["q_rows"].items():
            for d, v in row.items():
                q[int(i), 0, int(d)] = v
        inp = I.VerifyInputs(name=c["name"], q_lat=I.bf16_bits_from_f64(q[..., :dl]),
                             q_rope=I.bf16_bits_from_f64(q[..., dl:]),
                             kv_cache=I.bf16_bits_from_f64(kv),
                             block_table=np.zeros((1, 1), np.int32),
                             seq_lens=np.array([L], np.int32),
                             tree_parent=np.array(c["parent"], np.int32),
                             n_tree=np.array([T], np.int32), scale=c["scale"], page_size=L,
                             unique_pages=1)
        o, l = oracle.verify(inp, mutant=mutant)
        for i, (lse, outs) in enumerate(_hand_expect(c["name"], c["scale"])):
            assert abs(l[i, 0] - lse) < 1e-12, (c["name"], i)
            for d, v in outs.items():
                assert abs(o[i, 0, d] - v) < 1e-12, (c["name"], i, d)


def pin_validation(mutant=0):
    """Invalid trees and block ids are rejected with their status codes."""
    good = I.make_inputs([6], [4], tree_kind="uniform", page_size=2, seed=1, stream=13,
                         num_heads=1)
    assert oracle.check(good, mutant=mutant) == 0
    for par in ([-1, 1, 0, 0], [0, -1, 0, 1], [-1, 0, 3, 1], [-1, -2, 0, 0]):
        bad = I.VerifyInputs(**{**good.__dict__})
        bad.tree_parent = np.array(par, np.int32)
        assert oracle.check(bad, mutant=mutant) == 6
    bad = I.VerifyInputs(**{**good.__dict__})
    bad.block_table = good.block_table.copy()
    bad.block_table[0, 2] = good.num_pages
    assert oracle.check(bad, mutant=mutant) == 7


def _sparse_check(got, want, tol=1e-12):
    assert np.max(np.abs(got[0] - want[0])) <= tol and np.max(np.abs(got[1] - want[1])) <= tol


def pin_sparse_brute(mutant=0):
    """Sparse variant against the brute-force multiset definition (unused and repeated slots)."""
    from brute import brute_sparse
    for seed in range(3):
        inp = _tiny(seed, max_p=9)
        idx = I.topk_indices(inp, 6, seed=seed, unused_frac=0.25, duplicates=True)
        _sparse_check(oracle.verify_sparse(inp, idx, mutant=mutant), brute_sparse(inp, idx), 1e-11)


def pin_sparse_full_list_is_dense(mutant=0):
    """Listing every prefix position (any order, -1 padding) gives the dense result."""
    inp = _tiny(5, max_p=12)
    P = (inp.seq_lens - inp.n_tree).astype(int)
    topk = int(P.max()) + 3
    idx = I.topk_indices(inp, topk, seed=5)
    assert all(sorted(int(t) for t in idx[g] if t >= 0) == list(range(P[b]))
               for b in range(inp.batch) for g in range(int(inp.q_offsets[b]), int(inp.q_offsets[b + 1])))
    _sparse_check(oracle.verify_sparse(inp, idx, mutant=mutant), oracle.verify(inp, mutant=mutant))


def pin_sparse_repeated_slot_closed_form(mutant=0):
    """One root, slots [t, t]: weights 2e^{s_t} : e^{s_root}, so lse = ln(2e^{s_t} + e^{s_root})."""
    inp = I.make_inputs([7], [1], tree_kind="forest", page_size=2, seed=4, stream=20, num_heads=1)
    t = 3
    idx = np.array([[t, -1, t]], np.int32)
    out, lse = oracle.verify_sparse(inp, idx, mutant=mutant)
    from brute import logical_kv
    kv = logical_kv(inp, 0)
    q = np.concatenate([I.bf16_bits_to_f64(inp.q_lat[0, 0]), I.bf16_bits_to_f64(inp.q_rope[0, 0])])
    s_t = inp.scale * math.fsum(q * kv[t, :576])
    s_r = inp.scale * math.fsum(q * kv[7, :576])
    z = 2 * math.exp(s_t) + math.exp(s_r)
    assert abs(lse[0, 0] - math.log(z)) < 1e-12
    want = (2 * math.exp(s_t) * kv[t, :512] + math.exp(s_r) * kv[7, :512]) / z
    assert np.max(np.abs(out[0, 0] - want)) < 1e-12


def pin_sparse_validation(mutant=0):
    """A slot that is neither -1 nor a prefix position is rejected (status 9)."""
    inp = _tiny(6, max_p=9)
    P0 = int(inp.seq_lens[0] - inp.n_tree[0])
    for bad in (P0, -2, 1 << 20):
        idx = I.topk_indices(inp, 4, seed=6)
        idx[0, 1] = bad
        try:
            oracle.verify_sparse(inp, idx, mutant=mutant)
        except oracle.OracleError as e:
            assert e.status == 9
        else:
            raise AssertionError(f"slot {bad} accepted")


ALL_PINS = [pin_brute, pin_single_key, pin_uniform, pin_chain_causal, pin_split,
            pin_combine_closed_form, pin_permutation, pin_torch_library, pin_golden_hand,
            pin_validation, pin_sparse_brute, pin_sparse_full_list_is_dense,
            pin_sparse_repeated_slot_closed_form, pin_sparse_validation]
MUTANTS = {
    1: "rope term dropped from the score",
    2: "node does not see itself",
    3: "only the parent, not all ancestors, is visible",
    4: "softmax scale not applied",
    5: "lse returned in log2",
    6: "block table row of the wrong request",
    7: "weights not normalised",
    8: "V read at the wrong column offset",
    9: "tree keys shifted by one position",
    10: "combine uses the max instead of the log-sum-exp",
    11: "every listed top-k position off by one",
    12: "unused top-k slots attend to position 0",
}
