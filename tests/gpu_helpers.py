"""Shared helpers of the GPU parity tests (inputs, oracle calls, comparison rules)."""
import numpy as np

import oracle
from routed_expert_ffn_gemv_gb300 import synth

# Output tolerances: per-token max relative error (normwise, l-infinity) of layer
# outputs against the fp64 oracle; routes whose top-k margin is below GAP are excluded
# from the bit-exact id comparison.
TOL = 2e-3
GAP = 1e-5


def random_routes(rng, T, E, k):
    """Distinct expert ids per token and positive weights summing to 1."""
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.uniform(0.1, 1.0, size=(T, k))
    w = (w / w.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids, w


def ids_match(ids_gpu, logits_oracle, ids_oracle, k, gap=GAP):
    """Per token: True/False where comparable, None where the oracle's k-th/(k+1)-th margin < gap.

    Inside a selected list, positions whose adjacent oracle logits differ by < gap may
    appear in either order (compared as sets)."""
    out = []
    for t in range(ids_gpu.shape[0]):
        l = logits_oracle[t]
        order = np.lexsort((np.arange(l.size), -l))
        if k < l.size and l[order[k - 1]] - l[order[k]] < gap:
            out.append(None)
            continue
        ref = list(ids_oracle[t])
        got = list(ids_gpu[t])
        if set(ref) != set(got):
            out.append(False)
            continue
        ok = True
        i = 0
        while i < k:
            j = i
            while j + 1 < k and l[ref[j]] - l[ref[j + 1]] < gap:
                j += 1
            if set(ref[i:j + 1]) != set(got[i:j + 1]):
                ok = False
            i = j + 1
        out.append(ok)
    return out


def layer_oracle(cfg, layer, x64, route_override=None):
    wr = synth.router_weights(cfg, layer)
    b = synth.router_bias(cfg, layer)
    shared = [synth.expert_weights(cfg, layer, cfg.E + s) for s in range(cfg.n_shared)]
    return oracle.moe_layer(cfg.qtype, cfg.H, cfg.F, cfg.k, x64, wr, b,
                            lambda e: synth.expert_weights(cfg, layer, e), shared=shared,
                            route_override=route_override)


def rel_err(y, ref):
    return oracle.relative_error(y, ref)
