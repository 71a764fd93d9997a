"""Seeded synthetic inputs shared by the oracle and the CUDA path.

This module draws inputs only.  It holds none of the step's arithmetic
(no softmax, no selection, no cache, no expert FFN); the one computation it
does on router inputs is the tie-free conditioning described under
``tokens``.

Random streams: numpy PCG64 seeded with
``SeedSequence(seed, spawn_key=(cfg, kind, ...))``, so any single tensor (one
router, one expert, one token batch) can be drawn on its own.

Value recipes (the workload definition's, restated):
  * router weight Wr[E, d]: N(0, 0.02^2) rounded to bf16 (nearest, ties even);
  * activations x[T, d]: N(0, 1) rounded to bf16 (nearest, ties even);
  * packed expert weights: the 3-bit codes u = q + 4 are uniform on [0, 7],
    i.e. the packed code bytes are uniformly random bytes, so they are drawn
    as bytes; q = u - 4 is then uniform on [-4, 3];
  * group scales: U(0.005, 0.02) rounded to fp16 (nearest, ties even); the
    fp16 value is the definition;
  * stack router bias: per layer a seeded permutation gives each expert a
    Zipf rank r in 1..E and b = -lambda * s * ln(r) (fp32).

Canonical packed expert (what the host pool holds), in this order:
  Wg codes [f][d/32][12 B], Wu codes [f][d/32][12 B], Wd codes [d][f/32][12 B],
  Wg scales [f][d/32] fp16, Wu scales [f][d/32] fp16, Wd scales [d][f/32] fp16.
Within a 12-byte group, weight i (0..31, along the input dimension) is the
3-bit field at bits [3i, 3i+3) of the 96-bit little-endian integer.
"""

import numpy as np

from .configs import GROUP, MARGIN_DELTA, BIAS_LAMBDA, Workload, WORKLOADS, expert_nbytes

# stream kinds (part of the spawn key)
KIND_ROUTER_W = 1
KIND_ROUTER_PERM = 2
KIND_EXPERT = 3
KIND_SHARED = 4
KIND_X = 5
KIND_X_REDRAW = 6


def _rng(seed, *key):
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=tuple(int(k) for k in key))))


# ---------------------------------------------------------------- rounding --

def bf16_bits_from_f64(x):
    """Round float64 values to the nearest bf16 (ties to even); return the
    16-bit patterns.  Normal range only (|x| >= 2^-126 or x == 0)."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                       # x = m * 2^e, 0.5 <= |m| < 1
    r = np.rint(m * 256.0)                   # keep 8 significant bits
    v = np.ldexp(r, e - 8)
    nz = v != 0
    if np.any(np.abs(v[nz]) < 2.0 ** -126):
        raise ValueError("bf16 rounding: value below the normal range")
    return (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def bf16_bits_to_f64(bits):
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def fp16_from_f64(x):
    """Round float64 values to the nearest fp16 (ties to even), normal range."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    r = np.rint(m * 2048.0)                  # keep 11 significant bits
    v = np.ldexp(r, e - 11)
    nz = v != 0
    if np.any(np.abs(v[nz]) < 2.0 ** -14) or np.any(np.abs(v) > 65504.0):
        raise ValueError("fp16 rounding: value outside the normal range")
    return v.astype(np.float16)


# ------------------------------------------------------------------ layout --

def expert_sections(d, f, group=GROUP):
    """Byte offsets of the six sections of a canonical packed expert."""
    gq = f * (d // group) * 12
    dq = d * (f // group) * 12
    gs = f * (d // group) * 2
    ds = d * (f // group) * 2
    off = {}
    o = 0
    for name, n in (("wg_q", gq), ("wu_q", gq), ("wd_q", dq), ("wg_s", gs), ("wu_s", gs), ("wd_s", ds)):
        off[name] = (o, n)
        o += n
    assert o == expert_nbytes(d, f, group)
    return off


# ------------------------------------------------------------------ draws ---

class Synth:
    """Draws every input of one workload from its seed."""

    def __init__(self, wl: Workload, bias_lambda: float = BIAS_LAMBDA):
        self.wl = wl
        self.bias_lambda = bias_lambda
        self.B = expert_nbytes(wl.d, wl.f)
        self._router_cache = {}

    # router ---------------------------------------------------------------
    def router_weight_bits(self, layer):
        wl = self.wl
        rng = _rng(wl.seed, wl.cfg_id, KIND_ROUTER_W, layer)
        return bf16_bits_from_f64(rng.standard_normal((wl.n_experts, wl.d)) * 0.02)

    def router_bias(self, layer):
        """fp32 bias [E]; zeros unless the workload has a Zipf bias."""
        wl = self.wl
        if wl.zipf_s is None:
            return np.zeros(wl.n_experts, dtype=np.float32)
        rng = _rng(wl.seed, wl.cfg_id, KIND_ROUTER_PERM, layer)
        rank = rng.permutation(wl.n_experts) + 1
        return (-self.bias_lambda * wl.zipf_s * np.log(rank.astype(np.float64))).astype(np.float32)

    def router(self, layer):
        """(Wr bits [E,d] uint16, Wr as float64, bias fp32) for one layer, memoised."""
        r = self._router_cache.get(layer)
        if r is None:
            bits = self.router_weight_bits(layer)
            r = (bits, bf16_bits_to_f64(bits), self.router_bias(layer))
            self._router_cache[layer] = r
        return r

    # experts --------------------------------------------------------------
    def _packed(self, rng, out=None):
        wl = self.wl
        n = 3 * wl.d * wl.f
        nq = n * 3 // 8
        ns = n // GROUP
        if out is None:
            out = np.empty(self.B, dtype=np.uint8)
        out[:nq] = rng.integers(0, 256, size=nq, dtype=np.uint8)
        s = fp16_from_f64(0.005 + 0.015 * rng.random(ns))
        out[nq:] = s.view(np.uint8)
        return out

    def expert_packed(self, pool_index, out=None):
        """Canonical packed bytes of host-pool entry ``pool_index``."""
        wl = self.wl
        return self._packed(_rng(wl.seed, wl.cfg_id, KIND_EXPERT, pool_index), out)

    def shared_packed(self, layer, out=None):
        wl = self.wl
        return self._packed(_rng(wl.seed, wl.cfg_id, KIND_SHARED, layer), out)

    # tokens ---------------------------------------------------------------
    def _draw_x(self, rng, T):
        return bf16_bits_from_f64(rng.standard_normal((T, self.wl.d)))

    def tokens(self, layer, batch, T=None, stats=None):
        """Activations [T, d] (bf16 bits) for one call at one layer.

        Tie-free conditioning: the workload asks for router logits without
        ties, and bit-exact routing needs more than that, because the GPU
        computes logits in fp32 while the oracle uses fp64.  So a token is
        redrawn (from its own sub-stream) while the fp64 gap between its k-th
        and (k+1)-th largest logit x.Wr^T + b is below 1e-3, far above the
        ~1e-5 fp32 accumulation error at d=2048.  Only that gap is computed
        here; no routing decision is made.
        """
        return self.tokens_many(layer, [batch], T, stats)[0]

    def tokens_many(self, layer, batches, T=None, stats=None):
        """``tokens`` for several batch indices at one layer: [nb, T, d] bits."""
        wl = self.wl
        T = wl.tokens if T is None else T
        xs = np.empty((len(batches), T, wl.d), dtype=np.uint16)
        for i, b in enumerate(batches):
            xs[i] = self._draw_x(_rng(wl.seed, wl.cfg_id, KIND_X, layer, b), T)
        _, wr64, bias = self.router(layer)
        flat = xs.reshape(-1, wl.d)
        bad = self._small_gap(flat, wr64, bias)
        redraws = 0
        for idx in np.nonzero(bad)[0]:
            b = batches[idx // T]
            t = idx % T
            attempt = 0
            while True:
                cand = self._draw_x(_rng(wl.seed, wl.cfg_id, KIND_X_REDRAW, layer, b, t, attempt), 1)
                attempt += 1
                redraws += 1
                if not self._small_gap(cand, wr64, bias, exact=True)[0]:
                    flat[idx] = cand[0]
                    break
        if stats is not None:
            stats["redraws"] = stats.get("redraws", 0) + redraws
            stats["tokens"] = stats.get("tokens", 0) + flat.shape[0]
        return xs

    def _small_gap(self, xbits, wr64, bias, exact=False):
        """True where the fp64 gap between the k-th and (k+1)-th logit < delta.

        Large batches are screened in fp32 first; only tokens whose fp32 gap
        lies within 1e-4 of delta are re-evaluated in fp64, so the decision
        is the fp64 one.
        """
        k = self.wl.top_k
        x64 = bf16_bits_to_f64(xbits)
        if exact or x64.shape[0] <= 64:
            gap = _kth_gap(x64 @ wr64.T + bias.astype(np.float64), k)
            return gap < MARGIN_DELTA
        l32 = x64.astype(np.float32) @ wr64.astype(np.float32).T + bias
        gap32 = _kth_gap(l32.astype(np.float64), k)
        out = gap32 < MARGIN_DELTA
        unsure = np.nonzero(np.abs(gap32 - MARGIN_DELTA) < 1e-4)[0]
        if unsure.size:
            g = _kth_gap(x64[unsure] @ wr64.T + bias.astype(np.float64), k)
            out[unsure] = g < MARGIN_DELTA
        return out


def _kth_gap(logits, k):
    """Gap between the k-th and (k+1)-th largest value of each row."""
    E = logits.shape[1]
    part = np.partition(logits, (E - k - 1, E - k), axis=1)
    return part[:, E - k] - part[:, E - k - 1]


def synth(cfg_id, **kw):
    return Synth(WORKLOADS[cfg_id], **kw)
