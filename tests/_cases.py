"""Shared helpers of the parity tests: seeded cases, gap forcing, tolerances.

Inputs come from the seeded generator only; expected values come from the
CPU oracle only.
"""
from __future__ import annotations

import numpy as np

from mxfp4_routed_expert_k3_gb300 import synth
from mxfp4_routed_expert_k3_gb300.dims import LayerDims
from oracle import oracle as ora

GAP = 1e-3          # forced margin between the K-th and (K+1)-th router key
REL_RMS_TOL = 1e-2  # ||y - ref|| / ||ref||
MEAN_REL_TOL = 2e-3  # mean|y - ref| / mean|ref|
MAX_TOL = 1e-2      # |y_i - ref_i| <= MAX_TOL * rms(ref) + one bf16 ulp of ref_i
# routing weights: w = s / sum(s) moves by about (1 - s) * |d logit| for a
# logit error d logit.  fp32 sums on CUDA cores keep |d logit| ~ 1e-6; the
# tensor cores' fp32 accumulation drifts by up to ~K/16 * 2^-24 relative
# (K = 7168: ~3e-5, measured 3.4e-5), hence 5e-5.
W_RTOL = 5e-5


def gapped_tokens(d: LayerDims, w: dict, seed: int, T: int, max_attempts: int = 40) -> np.ndarray:
    """x [T, H] whose oracle keys have key_(K) - key_(K+1) > GAP for every
    token; offending rows are redrawn from the next attempt stream."""
    attempts = np.zeros(T, np.int64)
    x = synth.token_rows(d, seed, T)
    rows = np.arange(T)
    for _ in range(max_attempts):
        _, _, _, keys = ora.route(d, np.ascontiguousarray(x[rows]), w["router_w"], w["router_bias"],
                                  want_keys=True)
        gap = keys[:, d.top_k - 1].astype(np.float64) - keys[:, d.top_k].astype(np.float64)
        rows = rows[gap <= GAP]
        if rows.size == 0:
            return x
        attempts[rows] += 1
        for t in rows:
            synth.token_row_into(d, seed, int(t), int(attempts[t]), x[t])
    raise RuntimeError("could not force the routing gap")


def bf16_f64(bits) -> np.ndarray:
    return ora.bf16_to_float(np.asarray(bits).view(np.uint16) if np.asarray(bits).dtype != np.uint16 else bits)


def bf16_round(v: np.ndarray) -> np.ndarray:
    """float64 -> nearest bf16 value (as float64), through the oracle."""
    flat = np.asarray(v, np.float64).reshape(-1)
    bits = np.fromiter((ora.bf16_from_double(float(a)) for a in flat), dtype=np.uint16, count=flat.size)
    return ora.bf16_to_float(bits).reshape(np.shape(v))


_EXPERT_CACHE: dict = {}


def expert_matrix(w: dict, name: str, e: int) -> np.ndarray:
    """Expert e's w1 / w3 / w2 dequantised by the oracle, as float64."""
    key = (id(w), name, int(e))
    if key not in _EXPERT_CACHE or _EXPERT_CACHE[key][0] is not w:
        _EXPERT_CACHE[key] = (w, ora.bf16_to_float(ora.mxfp4_dequant_bf16(w[name + "_packed"][e],
                                                                          w[name + "_scale"][e])))
    return _EXPERT_CACHE[key][1]


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 7).astype(np.int64))


def y_metrics(y_bits, ref_bits, rounded_terms=()) -> dict:
    """Error figures of a bf16 output against the oracle's.  The per-element
    allowance is MAX_TOL * rms(ref) plus one bf16 ulp of ref and, when the
    output is the bf16 sum of separately rounded bf16 terms (the block with
    shared experts: y = bf16(y_routed + z)), one ulp of each such term:
    every rounded term may legitimately land one ulp from the oracle's."""
    g, r = bf16_f64(y_bits), bf16_f64(ref_bits)
    err = g - r
    rms = float(np.sqrt(np.mean(r * r)))
    allow = MAX_TOL * rms + bf16_ulp(r)
    for term in rounded_terms:
        allow = allow + bf16_ulp(np.asarray(term, np.float64))
    return {
        "rel_rms": float(np.sqrt(np.mean(err * err)) / rms),
        "mean_rel": float(np.mean(np.abs(err)) / np.mean(np.abs(r))),
        "max_over_rms": float(np.max(np.abs(err)) / rms),
        "max_excess": float(np.max(np.abs(err) - allow)),
        "identical_frac": float(np.mean(g == r)),
    }


def assert_y_close(y_bits, ref_bits, label="", rounded_terms=()):
    m = y_metrics(y_bits, ref_bits, rounded_terms)
    assert np.all(np.isfinite(bf16_f64(y_bits))), f"{label}: non-finite output"
    assert m["rel_rms"] <= REL_RMS_TOL, (label, m)
    assert m["mean_rel"] <= MEAN_REL_TOL, (label, m)
    assert m["max_excess"] <= 0.0, (label, m)
    return m


def assert_routing_equal(idx_gpu, w_gpu, idx_ref, w_ref, label=""):
    """Index sets must be identical per token; the order must be the
    descending-key order up to keys that fp32 cannot separate, so compare
    sorted sets, then the weights matched by expert id."""
    ig, ir = np.asarray(idx_gpu), np.asarray(idx_ref)
    assert ig.shape == ir.shape
    sg, sr = np.sort(ig, axis=1), np.sort(ir, axis=1)
    bad = np.flatnonzero(np.any(sg != sr, axis=1))
    assert bad.size == 0, f"{label}: index sets differ for tokens {bad[:10]}"
    og, orr = np.argsort(ig, axis=1), np.argsort(ir, axis=1)
    wg = np.take_along_axis(np.asarray(w_gpu, np.float64), og, 1)
    wr = np.take_along_axis(np.asarray(w_ref, np.float64), orr, 1)
    rel = np.abs(wg - wr) / np.maximum(np.abs(wr), 1e-30)
    worst = np.unravel_index(np.argmax(rel), rel.shape)
    assert np.allclose(wg, wr, rtol=W_RTOL, atol=1e-7), \
        f"{label}: routing weights differ: max rel {rel.max():.3e} at token {worst[0]} ({wg[worst]} vs {wr[worst]})"
    # order: the GPU lists experts in descending key order, like the oracle,
    # except possibly for neighbours whose fp32 keys coincide
    same_order = np.mean(np.all(ig == ir, axis=1))
    assert same_order > 0.95, f"{label}: order differs for {1 - same_order:.1%} of tokens"


def stable_permutation(idx: np.ndarray, E: int):
    """Reference grouping of the T*K assignments by expert (stable)."""
    flat = idx.reshape(-1)
    perm = np.argsort(flat, kind="stable").astype(np.int32)
    counts = np.bincount(flat, minlength=E).astype(np.int32)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    slot = np.empty_like(perm)
    slot[perm] = np.arange(perm.size, dtype=np.int32)
    return counts, offsets, perm, slot
