"""Independent brute-force evaluation of tree-verify attention for tiny inputs.

It shares nothing with the oracle's route to the answer: visibility comes from
a dense boolean transitive closure of the parent relation (Warshall), the
softmax is taken without a max shift, and every sum is an exactly rounded
``math.fsum``.  Only usable for a handful of keys per row.
"""
import math

import numpy as np

from mla_speculative_decoding_verify_gb300.inputs import bf16_bits_to_f64


def ancestor_matrix(parent):
    """A[i][j] is True iff j is i or an ancestor of i (Warshall closure)."""
    n = len(parent)
    A = [[i == j for j in range(n)] for i in range(n)]
    for i in range(n):
        if parent[i] >= 0:
            A[i][parent[i]] = True
    for k in range(n):
        for i in range(n):
            if A[i][k]:
                for j in range(n):
                    if A[k][j]:
                        A[i][j] = True
    return A


def logical_kv(inp, b):
    """Request b's KV rows in logical order, float64 [seq_len, 576]."""
    L = int(inp.seq_lens[b])
    rows = []
    for t in range(L):
        page = int(inp.block_table[b, t // inp.page_size])
        rows.append(inp.kv_cache[page, t % inp.page_size])
    return bf16_bits_to_f64(np.asarray(rows).reshape(L, -1))


def brute(inp, d_latent=512):
    H = inp.num_heads
    out = np.zeros((inp.total_q, H, d_latent))
    lse = np.zeros((inp.total_q, H))
    ql = bf16_bits_to_f64(inp.q_lat)
    qr = bf16_bits_to_f64(inp.q_rope)
    dr = qr.shape[-1]
    off = 0
    for b in range(inp.batch):
        T = int(inp.n_tree[b])
        P = int(inp.seq_lens[b]) - T
        par = [int(x) for x in inp.tree_parent[off:off + T]]
        A = ancestor_matrix(par)
        kv = logical_kv(inp, b)
        for i in range(T):
            vis = list(range(P)) + [P + j for j in range(T) if A[i][j]]
            for h in range(H):
                q = list(ql[off + i, h]) + list(qr[off + i, h])
                s = []
                for t in vis:
                    k = list(kv[t, :d_latent + dr])
                    s.append(inp.scale * math.fsum(a * c for a, c in zip(q, k)))
                e = [math.exp(x) for x in s]
                z = math.fsum(e)
                lse[off + i, h] = math.log(z)
                for d in range(d_latent):
                    out[off + i, h, d] = math.fsum(w * kv[t, d] for w, t in zip(e, vis)) / z
        off += T
    return out, lse


def brute_sparse(inp, topk_idx, d_latent=512):
    """Sparse variant: the visible multiset of tree token g is its listed prefix
    positions (one key per non-negative slot) plus its ancestor-or-self tree keys."""
    H = inp.num_heads
    out = np.zeros((inp.total_q, H, d_latent))
    lse = np.zeros((inp.total_q, H))
    ql = bf16_bits_to_f64(inp.q_lat)
    qr = bf16_bits_to_f64(inp.q_rope)
    dr = qr.shape[-1]
    off = 0
    for b in range(inp.batch):
        T = int(inp.n_tree[b])
        P = int(inp.seq_lens[b]) - T
        par = [int(x) for x in inp.tree_parent[off:off + T]]
        A = ancestor_matrix(par)
        kv = logical_kv(inp, b)
        for i in range(T):
            vis = [int(t) for t in topk_idx[off + i] if t >= 0] + [P + j for j in range(T) if A[i][j]]
            for h in range(H):
                q = list(ql[off + i, h]) + list(qr[off + i, h])
                s = [inp.scale * math.fsum(a * c for a, c in zip(q, list(kv[t, :d_latent + dr]))) for t in vis]
                e = [math.exp(x) for x in s]
                z = math.fsum(e)
                lse[off + i, h] = math.log(z)
                for d in range(d_latent):
                    out[off + i, h, d] = math.fsum(w * kv[t, d] for w, t in zip(e, vis)) / z
        off += T
    return out, lse

