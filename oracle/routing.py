"""Router: logits, softmax over all experts, top-k, renormalisation.

Structure from the pages: each token activates 10 of 512 routed experts per
layer plus one shared expert (P1 §如何做到：三层存储; P2 §1.3).  The formula is
the workload definition's: l = x.Wr^T + b; p = softmax(l) over all E; the
chosen set is the k largest logits (ties to the lower expert id); weights
w_i = p_i / sum_{j in set} p_j.  Indices are returned in ascending expert id,
a canonical order for the set.

Pins: brute force over all k-subsets on the tiny workload (the chosen set
maximises the sum of logits); renormalised weights equal a softmax over the
chosen logits alone; sum w = 1; k distinct ids; one-hot x selects a column
of Wr.
"""

import numpy as np


def router_logits(x, wr, bias=None):
    """x [T,d], wr [E,d] (exact bf16 values as fp64), bias [E] -> fp64 [T,E]."""
    l = np.asarray(x, np.float64) @ np.asarray(wr, np.float64).T
    if bias is not None:
        l = l + np.asarray(bias, np.float64)[None, :]
    return l


def softmax(l):
    """Row softmax in fp64 with the row maximum subtracted."""
    z = l - l.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def topk_ascending(l, k):
    """Ids of the k largest entries of each row (ties -> lower id), ascending."""
    T, E = l.shape
    out = np.empty((T, k), dtype=np.int64)
    ids = np.arange(E)
    for t in range(T):
        order = np.lexsort((ids, -l[t]))     # by value descending, then id ascending
        out[t] = np.sort(order[:k])
    return out


def route(x, wr, bias, k):
    """-> (idx [T,k] ascending expert id, w [T,k] fp64, logits [T,E])."""
    l = router_logits(x, wr, bias)
    p = softmax(l)
    idx = topk_ascending(l, k)
    pk = np.take_along_axis(p, idx, axis=1)
    w = pk / pk.sum(axis=1, keepdims=True)
    return idx, w, l
