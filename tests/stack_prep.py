"""Parallel preparation of a stack workload's inputs and oracle routing.

Each worker draws one layer's activations for every call of the stream and
routes them with the oracle.  The pool uses the 'spawn' start method so it
is safe to create after CUDA has been initialised.
"""

import concurrent.futures as cf
import multiprocessing as mp
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _layer_job(args):
    cfg_id, lam, layer, calls, overrides = args
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    from moe_inputs import Synth, WORKLOADS, bf16_bits_to_f64
    from oracle.routing import router_logits, softmax
    from oracle.stack import _route_rows
    import dataclasses
    wl = WORKLOADS[cfg_id]
    if overrides:
        wl = dataclasses.replace(wl, **overrides)
    s = Synth(wl, bias_lambda=lam)
    stats = {}
    xs = s.tokens_many(layer, list(range(calls)), stats=stats)
    _, wr64, b = s.router(layer)
    l = router_logits(bf16_bits_to_f64(xs.reshape(-1, wl.d)), wr64, b)
    p = softmax(l)
    idx = _route_rows(l, wl.top_k)
    pk = np.take_along_axis(p, idx, axis=1)
    w = pk / pk.sum(axis=1, keepdims=True)
    T = wl.tokens
    return layer, xs, idx.reshape(calls, T, wl.top_k), w.reshape(calls, T, wl.top_k), stats


def prepare_stack(cfg_id, lam, calls, n_layers, overrides=None, workers=None):
    """-> (x bits [L, calls, T, d], idx [L, calls, T, k], w [L, calls, T, k], redraw stats)."""
    workers = workers or min(16, os.cpu_count() or 1, n_layers)
    ctx = mp.get_context("spawn")
    out = [None] * n_layers
    stats = {"redraws": 0, "tokens": 0}
    with cf.ProcessPoolExecutor(max_workers=workers, mp_context=ctx) as ex:
        for layer, xs, idx, w, st in ex.map(_layer_job, [(cfg_id, lam, l, calls, overrides)
                                                          for l in range(n_layers)]):
            out[layer] = (xs, idx, w)
            stats["redraws"] += st.get("redraws", 0)
            stats["tokens"] += st.get("tokens", 0)
    xs = np.stack([o[0] for o in out])
    idx = np.stack([o[1] for o in out])
    w = np.stack([o[2] for o in out])
    return xs, idx, w, stats
