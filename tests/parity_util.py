"""Helpers shared by the GPU parity tests: oracle results on the same seeded
inputs, and the error metric.  Nothing here ever feeds a CUDA result into the
oracle."""
import os

import numpy as np

import oracle
from mxfp4_routed_expert_router_gb300 import workloads as wl

NTHREADS = max(1, min(32, os.cpu_count() or 1))

# max|gpu - oracle| / rms(oracle) on FP32 outputs (the layer's stated bound)
TOL = 1e-2
# routing weights: FP32 expf / division against the oracle's double
TOL_W = 1e-6


def rel_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    return float(np.max(np.abs(np.asarray(gpu, np.float64) - ref)) / rms)


def oracle_moe(cfg: wl.LayerConfig, x_bits: np.ndarray, logits: np.ndarray, tokens: np.ndarray, k: int = None):
    """Oracle output for the given token indices (their own x and logits rows)."""
    k = k or cfg.k
    xs, ls = x_bits[tokens], logits[tokens]
    ids, _ = oracle.route(ls, k)
    needed = sorted(set(ids.ravel().tolist()) | set(range(cfg.n_experts, cfg.n_groups)))
    W = oracle.OracleWeights(cfg.hidden, cfg.inter, cfg.n_experts, cfg.n_shared, cfg.weight_format)
    for e in needed:
        W.set_expert(e, *wl.expert_weights(cfg, e))
    out, ids, w = oracle.moe_layer(W, xs, ls, k, nthreads=NTHREADS)
    return out


def oracle_dense(cfg: wl.LayerConfig, x_bits: np.ndarray, tokens: np.ndarray, weights=None):
    weights = weights if weights is not None else wl.dense_weights(cfg)
    return oracle.dense_ffn(weights, x_bits[tokens], 0, cfg.weight_format)


def oracle_weights(cfg: wl.LayerConfig, experts) -> "oracle.OracleWeights":
    """Oracle weights holding the given experts (and every shared expert) of cfg."""
    W = oracle.OracleWeights(cfg.hidden, cfg.inter, cfg.n_experts, cfg.n_shared, cfg.weight_format)
    for e in sorted(set(int(v) for v in experts) | set(range(cfg.n_experts, cfg.n_groups))):
        W.set_expert(e, *wl.expert_weights(cfg, e))
    return W


def oracle_moe_routed(cfg: wl.LayerConfig, x_bits: np.ndarray, ids: np.ndarray, w: np.ndarray):
    """Oracle output of the layer for routing given as ids and weights (rows of x_bits)."""
    W = oracle_weights(cfg, np.unique(ids))
    return oracle.moe_layer_routed(W, x_bits, ids, w, nthreads=NTHREADS)


def skewed_logits(cfg: wl.LayerConfig, hot: int, n_hot: int, boost: float = 8.0) -> np.ndarray:
    """The config's logits with expert `hot` pushed to the top for the first
    n_hot tokens, so that one group holds many token tiles (a seeded test
    input; nothing of the layer's arithmetic)."""
    lg = wl.router_logits(cfg).copy()
    lg[:n_hot, hot] += np.float32(boost)
    return lg
