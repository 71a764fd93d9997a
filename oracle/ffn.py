"""Expert FFN (SwiGLU) and the routing-weighted combine, in fp64.

Structure from the pages: every token runs its 10 routed experts and one
shared expert per layer (P1 §如何做到：三层存储); all tokens of a verify batch
share one fetch of each expert (P2 §2.3).  The expert function is the
workload definition's SwiGLU, out = W_down . (silu(W_gate . x) * (W_up . x)),
silu(z) = z / (1 + e^-z); the layer output is
y[t] = sum_i w[t,i] * E_idx[t,i](x_t) + 1.0 * E_shared(x_t).

Pins: an explicit-loop formulation on the tiny workload; one-hot inputs pick
a column; identical experts make y independent of the routing; silu closed
forms; a dense matmul of the dequantised weights equals the group-wise
quantised dot products (brute force); a k-token batch equals k one-token
calls.
"""

import numpy as np


def silu(z):
    z = np.asarray(z, np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def expert_forward(W, x):
    """W = (Wg [f,d], Wu [f,d], Wd [d,f]); x [T,d] -> [T,d]."""
    wg, wu, wd = W
    g = x @ wg.T
    u = x @ wu.T
    h = silu(g) * u
    return h @ wd.T


def layer_forward(x, idx, w, expert_weights, shared_weights, shared_weight=1.0):
    """y [T,d] = sum_i w[t,i] E_idx[t,i](x_t) + shared_weight * E_shared(x_t).

    ``expert_weights(e)`` returns the fp64 matrices of routed expert e.
    Every distinct expert is evaluated once for all of its tokens.
    """
    x = np.asarray(x, np.float64)
    T = x.shape[0]
    y = shared_weight * expert_forward(shared_weights, x)
    for e in np.unique(idx):
        rows, cols = np.nonzero(idx == e)
        o = expert_forward(expert_weights(int(e)), x[rows])
        y[rows] += w[rows, cols][:, None] * o
    return y
