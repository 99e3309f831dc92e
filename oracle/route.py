"""Top-k routing: per-expert counts, segment offsets, inverse index, scatter.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Definition ("GEMM 执行方式", §4.2-§4.3 and §4.6; "AsymGEMM" README, "Token
Layout Protocols"):

* topk_ids[T, k_r] gives the expert of assignment (t, r); the flat index of
  an assignment is i = t * k_r + r.  Ids < 0 are dropped routes (§4.6 only
  scatters routes with expert_id >= 0); ids >= E are an error.
* M_e = number of assignments of expert e; with no drops sum_e M_e = T * k_r.
* Contiguous layout: expert e owns rows [seg_start[e], seg_start[e+1]) with
  seg_start[e+1] = seg_start[e] + ceil(M_e / A) * A (A = 1: unaligned §4.3;
  A = 128: the aligned layout of §4.6).  Rows past M_e inside a segment are
  padding.
* Masked layout: expert e owns rows [e * max_m, (e + 1) * max_m); at most
  max_m assignments are placed and the rest are dropped (reading: the pages
  give no overflow rule; here the later ones in flat order are dropped and
  counted).
* Order inside an expert (reading): ascending flat index, i.e. a stable sort
  by expert id.  §4.6 notes that an atomic scatter gives no fixed order; the
  worked example of §4.3 / §4.6 keeps token order, which is exactly this.
* output_index[t, r] = packed row of assignment (t, r), -1 if dropped;
  m_indices[row] = expert owning the row (padding rows included, as §4.6
  says); token_of_row[row] = token placed in the row, -1 for padding.

Pins: ``tests/test_oracle_route.py`` (the T=5, k_r=2, E=4 worked example of
§4.2-§4.6 from ``tests/golden/``, sum_e M_e = R, brute force on small random
inputs with duplicates and dropped ids, masked overflow).
"""

import numpy as np

CONTIGUOUS = 0
MASKED = 1


def route(topk_ids, num_experts, layout=CONTIGUOUS, align=1, max_m=0):
    """Compute the routing arrays; returns a dict of numpy arrays (see module doc)."""
    ids = np.asarray(topk_ids, dtype=np.int64)
    T, kr = ids.shape
    E = int(num_experts)
    flat = ids.reshape(-1)
    if np.any(flat >= E):
        raise ValueError("expert id >= number of experts")
    valid = flat >= 0
    M = np.bincount(flat[valid], minlength=E).astype(np.int64)

    # stable order by expert id: rank of each assignment among its expert's ones
    order = np.argsort(np.where(valid, flat, E), kind="stable")
    rank = np.empty(flat.size, dtype=np.int64)
    starts_sorted = np.concatenate([[0], np.cumsum(M)])
    for e in range(E):
        members = order[starts_sorted[e]:starts_sorted[e + 1]]
        rank[members] = np.arange(M[e])

    if layout == CONTIGUOUS:
        if align < 1:
            raise ValueError("align must be >= 1")
        seg_len = (M + align - 1) // align * align
        seg_start = np.concatenate([[0], np.cumsum(seg_len)]).astype(np.int64)
        placed = M.copy()
    elif layout == MASKED:
        if max_m < 1:
            raise ValueError("max_m must be >= 1")
        seg_start = np.arange(E + 1, dtype=np.int64) * max_m
        placed = np.minimum(M, max_m)
    else:
        raise ValueError("unknown layout")

    rows_used = int(seg_start[E])
    output_index = np.full(flat.size, -1, dtype=np.int64)
    token_of_row = np.full(rows_used, -1, dtype=np.int64)
    dropped = 0
    for i in range(flat.size):
        if not valid[i]:
            continue
        e = flat[i]
        if rank[i] >= placed[e]:
            dropped += 1
            continue
        row = seg_start[e] + rank[i]
        output_index[i] = row
        token_of_row[row] = i // kr

    m_indices = np.repeat(np.arange(E), np.diff(seg_start))
    return {
        "M": M,
        "counts": placed,
        "seg_start": seg_start,
        "output_index": output_index.reshape(T, kr),
        "token_of_row": token_of_row,
        "m_indices": m_indices,
        "rows_used": rows_used,
        "dropped": dropped,
    }


def scatter_rows(x, token_of_row, pad_value=0):
    """Packed copy of per-token rows: row r gets x[token_of_row[r]], padding rows pad_value."""
    x = np.asarray(x)
    out = np.full((len(token_of_row),) + x.shape[1:], pad_value, dtype=x.dtype)
    valid = token_of_row >= 0
    out[valid] = x[token_of_row[valid]]
    return out
