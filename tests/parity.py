"""Comparison rules of the GPU parity tests (the CUDA path against the oracle).

Tolerances: max |delta logit| <= 2e-2 over every compared row, and
final_norm_output relative L2 <= 1e-3 per row (f16 weights, f32
accumulation).  Greedy ids must be identical wherever the oracle's top-1
minus top-2 margin exceeds twice that row's max |delta logit| (capped at
2e-2); inside that margin either near-tied id is accepted.
"""
import numpy as np

LOGIT_TOL = 2e-2
HIDDEN_REL_L2 = 1e-3


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def top2_margin(row) -> float:
    r = np.asarray(row, dtype=np.float64)
    i = int(np.argmax(r.astype(np.float32)))
    rest = np.delete(r, i)
    return float(r[i] - rest.max())


def id_ok(gpu_id: int, orc_row, dl: float) -> bool:
    """Is ``gpu_id`` an accepted greedy pick for the oracle logits row?"""
    orc_row = np.asarray(orc_row, dtype=np.float64)
    orc_id = int(np.argmax(orc_row.astype(np.float32)))
    if gpu_id == orc_id:
        return True
    tie = min(2.0 * max(dl, 1e-6), LOGIT_TOL)
    return top2_margin(orc_row) <= tie and orc_row[gpu_id] >= orc_row[orc_id] - tie


def check_logits_ids(gpu_logits, gpu_ids, orc_logits, what: str = ""):
    gpu_logits = np.asarray(gpu_logits, dtype=np.float64).reshape(len(orc_logits), -1)
    orc_logits = np.asarray(orc_logits, dtype=np.float64).reshape(len(orc_logits), -1)
    d = np.abs(gpu_logits - orc_logits).max(axis=1)
    assert d.max() <= LOGIT_TOL, f"{what}: max |dlogit| {d.max():.3e} > {LOGIT_TOL}"
    for r in range(len(orc_logits)):
        assert id_ok(int(gpu_ids[r]), orc_logits[r], d[r]), \
            f"{what}: row {r} id {int(gpu_ids[r])} vs oracle {int(np.argmax(orc_logits[r]))} " \
            f"(margin {top2_margin(orc_logits[r]):.3e}, dl {d[r]:.3e})"
    return float(d.max())


def check_free_running(gpu_ids, orc_ids, orc_logits, what: str = "", dl: float = 1e-3):
    """Compare a free-running greedy id sequence with the oracle's; at the
    first difference the oracle's step must be a near-tie, after which the
    two sequences are no longer comparable.  Returns the steps compared."""
    gpu_ids = np.asarray(gpu_ids).reshape(-1)
    orc_ids = np.asarray(orc_ids).reshape(-1)
    for s in range(len(orc_ids)):
        if int(gpu_ids[s]) != int(orc_ids[s]):
            assert id_ok(int(gpu_ids[s]), orc_logits[s], dl), \
                f"{what}: step {s} id {int(gpu_ids[s])} vs oracle {int(orc_ids[s])} " \
                f"(margin {top2_margin(orc_logits[s]):.3e})"
            return s
    return len(orc_ids)


def check_hidden(gpu_h, orc_h, what: str = ""):
    gpu_h = np.asarray(gpu_h, dtype=np.float64).reshape(len(orc_h), -1)
    worst = max(rel_l2(gpu_h[r], orc_h[r]) for r in range(len(orc_h)))
    assert worst <= HIDDEN_REL_L2, f"{what}: hidden rel-L2 {worst:.3e} > {HIDDEN_REL_L2}"
    return worst


def check_kv(gpu_kv_seq, cache, positions, what: str = "", tol: float = 1e-3):
    """gpu_kv_seq: [L, 2, nkv, n_ctx, hd] of one sequence; cache: the
    oracle's KVCache.  Relative L2 per layer over the given positions."""
    pos = np.asarray(positions)
    for l in range(cache.K.shape[0]):
        gk = np.transpose(gpu_kv_seq[l, 0][:, pos], (1, 0, 2))
        gv = np.transpose(gpu_kv_seq[l, 1][:, pos], (1, 0, 2))
        ek = rel_l2(gk, cache.K[l, pos])
        ev = rel_l2(gv, cache.V[l, pos])
        assert ek <= tol and ev <= tol, f"{what}: layer {l} KV rel-L2 k {ek:.3e} v {ev:.3e}"
