"""Comparison rules of the GPU-vs-oracle parity tests.

Gate scores: within 1e-4 absolute (fp32 accumulation). Exit masks and
compaction indices: bit-exact, except tokens whose oracle score lies within
1e-3 of the threshold, which are excluded and counted. Filled K/V: max-abs
error at most 2e-2 and relative L2 error at most 1e-2 against the unrounded
float64 oracle.
"""
import numpy as np
import torch

SCORE_TOL = 1e-4
NEAR_BAND = 1e-3
KV_MAX_ABS = 2e-2
KV_REL_L2 = 1e-2


def f64(t) -> np.ndarray:
    if torch.is_tensor(t):
        return t.detach().double().cpu().numpy()
    return np.asarray(t, dtype=np.float64)


def host(x):
    """Layer dicts / tensors -> numpy (float64 for floating point, as-is for ints)."""
    if torch.is_tensor(x):
        return x.detach().double().cpu().numpy() if x.dtype.is_floating_point else x.detach().cpu().numpy()
    if isinstance(x, dict):
        return {k: host(v) for k, v in x.items()}
    if isinstance(x, (list, tuple)):
        return [host(v) for v in x]
    return x


def check_scores(gpu_score, ref_score):
    err = np.abs(f64(gpu_score) - ref_score)
    assert err.max(initial=0.0) <= SCORE_TOL, f"score error {err.max()}"


def check_mask(gpu_mask, ref_score, thr) -> int:
    """Mask bit-exact outside the near-threshold band; returns the excluded count."""
    ref = (ref_score.astype(np.float32) > np.float32(thr)).astype(np.uint8)
    near = np.abs(ref_score - thr) <= NEAR_BAND
    got = gpu_mask.cpu().numpy() if torch.is_tensor(gpu_mask) else gpu_mask
    bad = np.nonzero((got != ref) & ~near)[0]
    assert bad.size == 0, f"mask differs at {bad[:10]}"
    return int(near.sum())


def check_kv(gpu, ref, what="kv"):
    g = f64(gpu)
    diff = np.abs(g - ref)
    mx = diff.max(initial=0.0)
    rel = np.linalg.norm((g - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-30)
    assert mx <= KV_MAX_ABS and rel <= KV_REL_L2, f"{what}: max-abs {mx:.3e}, rel-L2 {rel:.3e}"
    return mx, rel


def check_decode_fill(cfg, x, rows, pos, seq, sentinel):
    """Written slots of a decode fill match the oracle; every other slot of both
    caches still holds ``sentinel``."""
    import oracle
    h = f64(x["h_cur"])
    layers = host(x["layers"])
    k_all, v_all = x["k_cache"], x["v_cache"]
    written = torch.zeros(k_all.shape[:4], dtype=torch.bool, device=k_all.device)
    dev = k_all.device
    for L in layers:
        if len(rows) == 0:
            break
        k_ref, v_ref = oracle.fill_rows(h[rows], L, pos[rows], cfg.n_kv_heads, cfg.head_dim, cfg.rope_base,
                                        cfg.eps, cfg.group)
        j = L["cache_layer"]
        idx_s = torch.as_tensor(seq[rows], device=dev).long()
        idx_p = torch.as_tensor(pos[rows], device=dev).long()
        check_kv(k_all[j, idx_s, :, idx_p], k_ref, f"K layer {j}")
        check_kv(v_all[j, idx_s, :, idx_p], v_ref, f"V layer {j}")
        written[j, idx_s, :, idx_p] = True
    for c in (k_all, v_all):
        assert bool((c[~written] == sentinel).all())
