"""Expert-parallel dispatch and combine: the rows one rank sends, in which
order, and how the results come back (oracle side; test infrastructure only).

The pages run the MoE layer with its experts spread over several GPUs and a
token all-to-all around the expert computation: DeepEP's all2all manager
(vLLM PR #35737, the CI failure logs: `all2all_manager.get_handle`, the
`deepep_high_throughput` prepare/finalize of the MoE layer, and DeepEP's
buffer set-up through torch.distributed).  They show the call sites, not the
data layout.  Readings (each listed in the design notes):

  * G ranks each hold T_r tokens (data parallel) and route them over all E
    routed experts; rank r owns routed experts [r E/G, (r+1) E/G) (E/G local
    experts, E a multiple of G); a shared expert is replicated: every rank
    computes its own tokens' shared rows, as local expert E/G;
  * dispatch after quantization: a rank sends each (token, slot) assignment's
    NVFP4 A1 row (quantized with the destination expert's activation global
    scale) to the expert's owner; the rows for rank r are the rank's
    permutation (stable by expert, then assignment index) restricted to r's
    experts, in that order; the rank's own segment ends with its shared rows
    (by token);
  * the receiver groups the rows by local expert: expert j's rows are source
    0's rows of j, then source 1's, ... (each in arrival order);
  * each y row returns to its sender at the position it was sent from, and the
    sender combines exactly as without expert parallelism.

The expert computation of a row does not depend on which other rows share its
expert, so every rank's output equals the single-device forward of its own
tokens; the pins check exactly that, plus brute-force counts and the
bijectivity of the plan.
"""
from __future__ import annotations

import numpy as np

from . import formats as F
from . import moe as M

F32 = np.float32


def owner(e: int, E: int, G: int) -> int:
    """Rank owning routed expert e (contiguous blocks of E/G experts)."""
    return int(e) // (E // G)


def dispatch_plan(ids, E: int, G: int, rank: int, shared: bool):
    """Rows one rank sends.  ids: [T, k] routed expert ids of the rank's tokens.

    Returns (segments, counts, src_to_send):
      segments[r]    list of (assignment a, global expert e) in send order to
                     rank r (a = t*k + j for routed rows, T*k + t for shared rows);
      counts[r, j]   rows for local expert j of rank r (j = E/G: the shared
                     expert, nonzero only for r == rank);
      src_to_send[a] position of assignment a in the concatenated send buffer
                     (segments of ranks 0..G-1 back to back).
    """
    ids = np.asarray(ids)
    T, k = ids.shape
    El = E // G
    counts_e, offsets, p2s, _ = M.permute(ids, E, shared)
    segments = [[] for _ in range(G)]
    for p, a in enumerate(p2s):                       # permuted order: by expert, then by assignment
        a = int(a)
        e = int(ids.reshape(-1)[a]) if a < T * k else E
        dest = owner(e, E, G) if e < E else rank
        segments[dest].append((a, e))
    counts = np.zeros((G, El + 1), np.int64)
    for r in range(G):
        for a, e in segments[r]:
            counts[r, e - r * El if e < E else El] += 1
    src_to_send = np.full(T * k + (T if shared else 0), -1, np.int64)
    pos = 0
    for r in range(G):
        for a, _ in segments[r]:
            src_to_send[a] = pos
            pos += 1
    return segments, counts, src_to_send


def receive_order(counts_in):
    """Grouped order on a receiving rank.  counts_in: [G, El+1] rows per local
    expert arriving from each source (the sources' counts[r]).  Returns
    (local_offsets [El+2], recv_to_grp [n]): received row i (sources back to
    back, each source's rows by local expert) goes to grouped row
    recv_to_grp[i]; local expert j's grouped rows are source 0's, source 1's, ..."""
    counts_in = np.asarray(counts_in, np.int64)
    G, J = counts_in.shape
    per_expert = counts_in.sum(axis=0)
    local_offsets = np.concatenate([[0], np.cumsum(per_expert)])
    recv_to_grp = []
    for s in range(G):
        for j in range(J):
            start = local_offsets[j] + counts_in[:s, j].sum()
            recv_to_grp.extend(range(int(start), int(start + counts_in[s, j])))
    return local_offsets, np.array(recv_to_grp, np.int64)


def ep_forward(xs, logits, k: int, E: int, G: int, shared: bool, renormalize: bool, weights, gs_a1, gs_a2):
    """The layer over G ranks with expert parallelism.  xs[r]: float32 [T_r, H]
    tokens of rank r, logits[r]: [T_r, E]; weights(e) and gs_a1/gs_a2 [E'] as
    in moe.moe_forward (global expert ids).  Returns per rank a dict with
    out [T_r, H] (float64) and the plan (segments, counts, src_to_send),
    plus per receiving rank the grouped order."""
    El = E // G
    H = np.asarray(xs[0]).shape[1]
    plans = []
    for r in range(G):
        ids, w = M.route(logits[r], None, k, renormalize)
        segs, counts, s2s = dispatch_plan(ids, E, G, r, shared)
        plans.append(dict(ids=ids, weights=w, segments=segs, counts=counts, src_to_send=s2s))
    # each receiver: rows from every source, grouped by local expert
    y_back = [np.full((len(p["src_to_send"]), H), np.nan) for p in plans]
    recv = []
    for r in range(G):
        counts_in = np.stack([plans[s]["counts"][r] for s in range(G)])
        loc_off, r2g = receive_order(counts_in)
        arrivals = [(s, i, a, e) for s in range(G) for i, (a, e) in enumerate(plans[s]["segments"][r])]
        grouped = [None] * len(arrivals)
        for n, item in enumerate(arrivals):
            grouped[r2g[n]] = item
        recv.append(dict(counts_in=counts_in, local_offsets=loc_off, recv_to_grp=r2g))
        # the expert computation, one local expert's grouped rows at a time
        for j in range(El + (1 if shared else 0)):
            rows = grouped[loc_off[j]:loc_off[j + 1]]
            if not rows:
                continue
            e = r * El + j if j < El else E
            T_src = [len(xs[s]) for s in range(G)]
            xr = np.stack([np.asarray(xs[s], F32)[M.assignment_token(np.array([a]), T_src[s], k)[0]]
                           for s, _, a, _ in rows])
            w13c, w13s, gw13, w2c, w2s, gw2 = weights(e)
            I = w13c.shape[0] // 2
            ac, asc = F.quantize_rows(xr, gs_a1[e])
            c1 = np.float64(M.alpha(gs_a1[e], gw13)) * M.block_scaled_matmul(ac, asc, w13c, w13s)
            h = M.swiglu(c1, I).astype(F32)
            qc, qs = F.quantize_rows(h, gs_a2[e])
            y = np.float64(M.alpha(gs_a2[e], gw2)) * M.block_scaled_matmul(qc, qs, w2c, w2s)
            # back to the sender, at the position the row was sent from
            for (s, _, a, _), yr in zip(rows, y):
                y_back[s][plans[s]["src_to_send"][a]] = yr
    outs = []
    for r in range(G):
        T = len(xs[r])
        out = M.combine(y_back[r], plans[r]["weights"], plans[r]["src_to_send"], T, k, shared)
        outs.append(dict(out=out, y_back=y_back[r], **plans[r]))
    return outs, recv
