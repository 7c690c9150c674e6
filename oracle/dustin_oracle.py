"""fp64 CPU oracle of the Dustin sparse-verification hot path.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import or call this module.  The product
path (the CUDA library and its Python binding) never does, and this module
imports nothing from it.

Every function restates one step of the method as the Dustin pages describe
it ("Technical Summary: Dustin", gist.science/paper/2606.24957, sections
"1. Hybrid Attention Aggregation", "2. Efficient Estimation via Semantic
Retrieval Heads (SRHs)" and "3. Verification Workflow"), plainly and slowly:
bf16 inputs are widened exactly to float64, ``np.exp`` runs in float64, and no
step is blocked, fused or reordered.  Where the pages leave a step open, the
reading taken is named in the docstring (R1..R15 are the numbered readings
listed in the design notes).

Inputs are host ``uint16`` arrays of bf16 bit patterns (see ``bf16``).
"""
from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------


def bf16(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) exactly to float64."""
    b = np.asarray(bits)
    if b.dtype != np.uint16:
        raise TypeError("expected uint16 bf16 bit patterns")
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def softmax(x: np.ndarray, axis: int = -1) -> np.ndarray:
    """Textbook softmax with max subtraction, in float64."""
    m = np.max(x, axis=axis, keepdims=True)
    e = np.exp(x - m)
    return e / np.sum(e, axis=axis, keepdims=True)


def kv_group(h: int, hq: int, hkv: int) -> int:
    """KV head read by query head ``h`` under grouped-query attention.

    Reading R4: contiguous groups, ``g = h // (hq / hkv)`` (the Qwen2.5 layout;
    the pages do not say).
    """
    return h // (hq // hkv)


# ---------------------------------------------------------------------------
# 1. hybrid importance scoring on SRHs
# ---------------------------------------------------------------------------


def score(draft_q, Kd, hist_q, K, srh, seq_len, Lcap):
    """Global importance map ``imp[B][2][Lcap]`` (float64).

    Follows "1. Hybrid Attention Aggregation" (target-historical and
    draft-look-ahead attention scores aggregated into one global importance
    map) restricted, as "2. Efficient Estimation via SRHs" says, to the SRH
    heads only.

    ``srh`` lists ``(channel, layer, q_head)``.  Channel 0 is the draft
    look-ahead signal: queries ``draft_q[layer][b, :, h]`` (gamma rows) against
    the draft cache ``Kd[layer]``.  Channel 1 is the target historical signal:
    queries ``hist_q[layer][b, :, h]`` (gamma+1 rows) against the target cache
    ``K[layer]``.

    For each SRH and each of its query rows (a "pair") the attention
    probabilities over the ``L = seq_len[b]`` context positions are
    ``softmax_i(q . k_i / sqrt(d))`` (readings R1 post-softmax scores, R3
    1/sqrt(d) scale, R5 no causal mask inside the context), and the map is
    their plain sum over pairs within each channel (reading R2).  Positions at
    or beyond ``L`` stay 0.
    """
    B = len(seq_len)
    imp = np.zeros((B, 2, Lcap), dtype=np.float64)
    for (channel, layer, h) in srh:
        qs = draft_q[layer] if channel == 0 else hist_q[layer]
        cache = Kd[layer] if channel == 0 else K[layer]
        hq, hkv, d = qs.shape[2], cache.shape[1], cache.shape[3]
        g = kv_group(h, hq, hkv)
        for b in range(B):
            L = int(seq_len[b])
            if L == 0:
                continue
            keys = bf16(cache[b, g, :L, :])            # [L][d]
            for t in range(qs.shape[1]):
                q = bf16(qs[b, t, h, :])               # [d]
                logits = keys @ q / math.sqrt(d)        # [L]
                imp[b, channel, :L] += softmax(logits)
    return imp


# ---------------------------------------------------------------------------
# 2. budgeted tiered selection of I_verify
# ---------------------------------------------------------------------------


def protected_sets(L: int, sinks: int, window: int):
    """Sink prefix and recent window (reading R7: their union, counted once)."""
    s_eff = min(sinks, L)
    w0 = max(L - window, s_eff)
    return np.arange(0, s_eff), np.arange(w0, L)


def _top_by(scores: np.ndarray, cand: np.ndarray, n: int) -> np.ndarray:
    """First ``n`` candidates ordered by (score descending, index ascending).

    Reading R8: equal scores go to the lower position first.
    """
    if n <= 0:
        return np.zeros(0, dtype=np.int64)
    order = np.lexsort((cand, -scores[cand]))
    return np.sort(cand[order[:n]])


def select(imp, seq_len, k, sinks, window, m):
    """Fixed-size verification set ``I_verify[B][k]`` (int64) and tier sizes.

    Follows "1. Hybrid Attention Aggregation": protect a sink prefix and a
    recent window, fill the rest of a fixed budget of ``k`` with the top-``m``
    positions by the draft signal (channel 0) and then the most relevant
    remaining positions by the target signal (channel 1).

    Readings: R6 the sinks and the window count inside ``k``; R7 if
    ``k >= L`` every context position is taken, in ascending order, and the
    tail is padded with -1; R8 ties go to the lower index; R12 the output is
    four ascending segments ``[sinks | window | draft tier | target tier]``.
    Returns ``(I, tiers)`` with ``tiers[b] = (n_sinks, n_window, m', f)``.
    """
    B = len(seq_len)
    out = np.full((B, k), -1, dtype=np.int64)
    tiers = []
    for b in range(B):
        L = int(seq_len[b])
        if k >= L:
            out[b, :L] = np.arange(L)
            tiers.append((L, 0, 0, 0))
            continue
        sink_part, win_part = protected_sets(L, sinks, window)
        n_p = sink_part.size + win_part.size
        if n_p > k:
            raise ValueError("protected set larger than the budget")
        U = np.arange(sink_part.size, win_part[0] if win_part.size else L)
        m1 = min(m, k - n_p)
        f = k - n_p - m1
        D = _top_by(imp[b, 0], U, m1)
        rest = np.setdiff1d(U, D)
        R = _top_by(imp[b, 1], rest, f)
        out[b] = np.concatenate([sink_part, win_part, D, R])
        tiers.append((sink_part.size, win_part.size, m1, f))
    return out, tiers


# ---------------------------------------------------------------------------
# 3. sparse verification attention (and the dense comparator)
# ---------------------------------------------------------------------------


def _attend(Q, K, V, Kb, Vb, rows_of_b):
    """Shared definition for sparse and dense verification.

    For sequence ``b``, verify query ``t`` (0..gamma) of head ``h`` (KV head
    ``g``) attends to the cache rows ``rows_of_b(b)`` plus the draft-block
    rows ``u <= t`` (reading R9: causal inside the block), with softmax
    weights of ``q . k / sqrt(d)``; the output is the weighted sum of values.
    """
    B, T, hq, d = Q.shape
    hkv = K.shape[1]
    O = np.zeros((B, T, hq, d), dtype=np.float64)
    for b in range(B):
        rows = rows_of_b(b)
        for g in range(hkv):
            kc = bf16(K[b, g, rows, :])
            vc = bf16(V[b, g, rows, :])
            kb = bf16(Kb[b, g])
            vb = bf16(Vb[b, g])
            for h in range(hq):
                if kv_group(h, hq, hkv) != g:
                    continue
                for t in range(T):
                    keys = np.concatenate([kc, kb[: t + 1]])
                    vals = np.concatenate([vc, vb[: t + 1]])
                    q = bf16(Q[b, t, h, :])
                    p = softmax(keys @ q / math.sqrt(d))
                    O[b, t, h, :] = p @ vals
    return O


def verify(Q, K, V, Kb, Vb, I, seq_len):
    """Sparse verification attention, float64 ``O[B][gamma+1][Hq][d]``.

    Follows "3. Verification Workflow", steps 3-4: a compressed target cache
    made of the top-k selected rows, and verification of the draft tokens
    against it.  Reading R11: the compressed cache is the rows ``I[b]`` of the
    full cache (no copy); entries -1 are padding and are skipped.
    """
    def rows(b):
        r = np.asarray(I[b])
        r = r[r >= 0]
        if np.any(r >= int(seq_len[b])):
            raise ValueError("index beyond the context")
        return r
    return _attend(Q, K, V, Kb, Vb, rows)


def dense(Q, K, V, Kb, Vb, seq_len):
    """Full-cache verification, the comparator ("Problem Statement": standard
    speculative decoding loads the whole KV cache to verify the draft)."""
    return _attend(Q, K, V, Kb, Vb, lambda b: np.arange(int(seq_len[b])))


# ---------------------------------------------------------------------------
# 4. append accepted tokens
# ---------------------------------------------------------------------------


def kv_append(K, V, Kb, Vb, n_accept, seq_len):
    """Cache after appending the accepted draft rows ("3. Verification
    Workflow", step 5: accepted tokens are appended to the cache, rejected ones
    discarded).  Returns new ``(K, V, seq_len)``; inputs are not modified."""
    K2, V2 = K.copy(), V.copy()
    sl = np.array(seq_len, dtype=np.int64).copy()
    for b in range(K.shape[0]):
        n = int(n_accept[b])
        L = int(sl[b])
        K2[b, :, L:L + n, :] = Kb[b, :, :n, :]
        V2[b, :, L:L + n, :] = Vb[b, :, :n, :]
        sl[b] = L + n
    return K2, V2, sl.astype(np.int32)


# ---------------------------------------------------------------------------
# quality report: attention recovery
# ---------------------------------------------------------------------------


def attention_recovery(Q, K, I, seq_len):
    """Fraction of dense verification attention mass that falls on ``I``.

    Reading R14 of the "Attention Recovery Rate" that "2. Efficient Estimation
    via SRHs" names as the offline objective: for every verify query and head,
    the dense softmax over the context is taken and the mass on the selected
    rows summed; the mean over queries and heads is reported per sequence.
    """
    B, T, hq, d = Q.shape
    hkv = K.shape[1]
    arr = np.zeros(B)
    for b in range(B):
        L = int(seq_len[b])
        sel = np.asarray(I[b])
        sel = sel[sel >= 0]
        tot = 0.0
        for h in range(hq):
            keys = bf16(K[b, kv_group(h, hq, hkv), :L, :])
            for t in range(T):
                p = softmax(keys @ bf16(Q[b, t, h, :]) / math.sqrt(d))
                tot += p[sel].sum()
        arr[b] = tot / (hq * T)
    return arr
