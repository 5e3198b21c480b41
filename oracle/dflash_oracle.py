"""fp64 CPU oracle for the DFlash draft body, its batch plan and greedy verification.

TEST INFRASTRUCTURE ONLY.  This module is the slow, plain definition the CUDA library is
checked against.  Only the tests, the smoke check and the benchmark's CPU-baseline /
reference arms may import it; the library never calls it and shares no code with it.

Sources (the three DFlash pages; cited by page title and section):
* "DFlash" (angelspec docs) -- "How it works": block-parallel prediction with a
  block-causal mask, dual-source K/V (target hidden states projected by W_proj),
  anchor sampling; "Configuration": target_layer_ids, rope_theta.
* "DFlash Draft Body" (NeMo RL design doc) -- "How It Works" steps 1-4: deterministic
  anchor plan from (mask, sample ids, step, seed), same sample id => same anchors, a block
  reads the target prefix before its anchor plus its own block and never another block,
  one hidden state per block position with zeros at invalid positions, loss_mask excludes
  the anchor and invalid positions.
* "DFlash: drafting, verification, and speed" -- "One DFlash generation cycle" (greedy
  verification: longest matching prefix, the target's correction at the first mismatch,
  the bonus token when all proposals match, optional EOS stop; the information boundary).

Where the pages leave a step open, the reading used is stated at the function.  The
readings are numbered R1..R12 and are the same ones the CUDA library implements.

Everything floating point is float64 with no intermediate rounding.  Integer work (the
plan, argmax indices, verification) is exact Python/NumPy integer arithmetic.

Parity pins: every function here is pinned by tests under tests/ (test_oracle_*.py)
against closed forms, brute force, invariants or the pages' worked example.  The one
exception is the anchor-key hash constant set: it is this library's own definition (the
pages fix none); it is pinned to the published SplitMix64 reference outputs and fixed by
golden vectors (tests/golden/plan_*.txt).
"""
from __future__ import annotations

import math

import numpy as np

U64 = (1 << 64) - 1

# ======================================================================================
# Plan (anchor sampling, block membership, loss mask)
# ======================================================================================


def splitmix64_mix(z: int) -> int:
    """SplitMix64 output finaliser (Steele, Lea & Flood, "Fast splittable pseudorandom
    number generators", OOPSLA 2014; the variant with shifts 30/27/31) on uint64."""
    z &= U64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & U64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & U64
    return z ^ (z >> 31)


def splitmix64_stream(seed: int, n: int) -> list:
    """The SplitMix64 generator itself (state advanced by the golden gamma before each
    finalisation).  Used only to pin splitmix64_mix against published reference outputs."""
    out, s = [], seed & U64
    for _ in range(n):
        s = (s + 0x9E3779B97F4A7C15) & U64
        out.append(splitmix64_mix(s))
    return out


def anchor_key(seed: int, step: int, sample_id: int, pos: int) -> int:
    """R3: the sort key of candidate anchor `pos` in a row with sample id `sample_id`.

    "DFlash Draft Body", How It Works step 1 fixes only that the plan is a function of
    (input mask, sample ids, optimizer step, seed).  This library's definition: a chained
    SplitMix64 finaliser over the four values, each taken as uint64 (two's complement)."""
    h = splitmix64_mix(seed & U64)
    h = splitmix64_mix(h ^ (step & U64))
    h = splitmix64_mix(h ^ (sample_id & U64))
    return splitmix64_mix(h ^ (pos & U64))


def _valid(mask_row, p: int) -> bool:
    return 0 <= p < len(mask_row) and mask_row[p] != 0


def anchor_candidates(mask_row) -> list:
    """R2: position a can anchor a block iff a is valid and a + 1 is valid, i.e. the block
    has at least one position to predict ("a sample with no valid window contributes no
    draft loss", "DFlash Draft Body", How It Works step 1).  Blocks may run past the valid
    end; those tail slots are invalid."""
    return [a for a in range(len(mask_row)) if _valid(mask_row, a) and _valid(mask_row, a + 1)]


def choose_anchors(mask_row, sample_id: int, step: int, seed: int, num_anchors: int) -> list:
    """R3: uniform sampling without replacement, made deterministic: the num_anchors
    candidates with the smallest (key, position) pairs, returned in increasing position.
    Fewer candidates than num_anchors: all of them, the remaining slots are -1."""
    cands = anchor_candidates(mask_row)
    keyed = sorted((anchor_key(seed, step, sample_id, a), a) for a in cands)
    chosen = sorted(a for _, a in keyed[:num_anchors])
    return chosen + [-1] * (num_anchors - len(chosen))


def build_plan(mask, sample_ids, step: int, seed: int, num_anchors: int, block_size: int):
    """The batch plan ("DFlash Draft Body", How It Works steps 1, 2 and 4).

    mask [B, L] (nonzero = valid), sample_ids [B] int.  Returns a dict of int arrays:
      anchors      [B, N]    int32, sorted valid anchors then -1
      block_valid  [B, N, S] uint8  (R5)
      loss_mask    [B, N, S] uint8  block_valid and slot j >= 1 (the anchor never counts)
      position_ids [B, N, S] int32  anchor + j (R1), -1 for empty slots

    R4 ("rows with the same sample ID get the same anchors"): the lowest-index row with a
    given sample id draws the anchors from its own mask; every row with that id takes the
    same anchor list.  Validity and the loss mask come from each row's own mask."""
    mask = np.asarray(mask)
    B, L = mask.shape
    N, S = num_anchors, block_size
    anchors = np.full((B, N), -1, np.int32)
    block_valid = np.zeros((B, N, S), np.uint8)
    position_ids = np.full((B, N, S), -1, np.int32)
    sids = [int(x) for x in np.asarray(sample_ids).reshape(-1)]
    leader_list = {}
    for b in range(B):
        if sids[b] not in leader_list:
            leader_list[sids[b]] = choose_anchors(list(mask[b]), sids[b], step, seed, N)
        anchors[b] = leader_list[sids[b]]
    for b in range(B):
        row = list(mask[b])
        for k in range(N):
            a = int(anchors[b, k])
            if a < 0:
                continue
            for j in range(S):
                position_ids[b, k, j] = a + j
                block_valid[b, k, j] = 1 if (_valid(row, a) and _valid(row, a + j)) else 0
    loss_mask = block_valid.copy()
    loss_mask[:, :, 0] = 0
    return {"anchors": anchors, "block_valid": block_valid, "loss_mask": loss_mask,
            "position_ids": position_ids}


# ======================================================================================
# Layer arithmetic (textbook definitions)
# ======================================================================================


def rms_norm(x: np.ndarray, gain: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * gain."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * gain


def rope_angles(positions: np.ndarray, head_dim: int, theta: float) -> np.ndarray:
    """R7: angle[p, i] = position_p * theta^(-2i/dh), i < dh/2 (fp64)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / head_dim)
    return np.asarray(positions, np.float64)[:, None] * inv_freq[None, :]


def apply_rope(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """R7 rotate-half RoPE: x [P, H, dh], one position per leading index.
    Channel i is paired with channel i + dh/2 and the pair is rotated by angle[p, i]."""
    dh = x.shape[-1]
    half = dh // 2
    ang = rope_angles(positions, dh, theta)[:, None, :]
    c, s = np.cos(ang), np.sin(ang)
    lo, hi = x[..., :half], x[..., half:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def softmax_rows(s: np.ndarray) -> np.ndarray:
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


# ======================================================================================
# Context projection (dual-source K/V, the target-side half)
# ======================================================================================


def project_context_row(cfg, top, layers, hidden_row: np.ndarray, positions=None):
    """Context K/V for one batch row (R8).

    "DFlash", How it works (Dual-source KV context): the target's selected multi-layer
    hidden states are projected by W_proj and attended alongside the draft tokens' own
    K/V.  Reading R8: ctx = RMSNorm(H_cat W_proj^T; g_ctx) (norm switchable by
    cfg.ctx_norm); each draft layer l enters its own K/V space through its own key/value
    projections: K_ctx = RoPE(ctx W_k^T) at position c, V_ctx = ctx W_v^T.

    hidden_row [P, n_tl*D_t] fp64 (positions 0..P-1 unless `positions` given);
    top = {w_proj [D, n_tl*D_t], g_ctx [D]}; layers: callable l -> layer dict.
    Returns a list over layers of (K [Hkv, P, dh], V [Hkv, P, dh])."""
    P = hidden_row.shape[0]
    pos = np.arange(P) if positions is None else np.asarray(positions)
    y = hidden_row @ top["w_proj"].T
    ctx = rms_norm(y, top["g_ctx"], cfg.rms_eps) if cfg.ctx_norm else y
    qw, kw = cfg.num_heads * cfg.head_dim, cfg.num_kv_heads * cfg.head_dim
    out = []
    for l in range(cfg.num_layers):
        w_qkv = layers(l)["w_qkv"]
        k = (ctx @ w_qkv[qw:qw + kw].T).reshape(P, cfg.num_kv_heads, cfg.head_dim)
        v = (ctx @ w_qkv[qw + kw:qw + 2 * kw].T).reshape(P, cfg.num_kv_heads, cfg.head_dim)
        k = apply_rope(k, pos, cfg.rope_theta)
        out.append((np.transpose(k, (1, 0, 2)), np.transpose(v, (1, 0, 2))))
    return out


def commit_verified(cache_hidden: np.ndarray, verified_hidden: np.ndarray,
                    accepted: int) -> np.ndarray:
    """Cache rollback after greedy verification ("DFlash: drafting, verification, and
    speed", One DFlash generation cycle, the paragraph after the worked example).

    The target's verification pass computes states for every position of the block -- the
    anchor and all gamma proposals -- but only the verified prefix may stay in a cache:
    the anchor and the `accepted` proposals that matched.  The rejected proposal and its
    suffix are dropped; the target's replacement token (or the bonus) has had no forward
    pass yet and becomes the anchor of the next block, at the position right after the
    retained prefix.  The draft's context cache must stay aligned with the target's, so it
    retains the same positions.

    cache_hidden [P0, W]: committed hidden states so far (positions 0 .. P0-1);
    verified_hidden [S, W]: the block's states (anchor first), S = gamma + 1;
    accepted: proposals accepted (0 .. gamma).  Returns the committed states [P0 + accepted
    + 1, W]; the next block is anchored at position P0 + accepted + 1."""
    S = verified_hidden.shape[0]
    if not 0 <= accepted <= S - 1:
        raise ValueError("accepted must lie in [0, gamma]")
    return np.concatenate([cache_hidden, verified_hidden[:accepted + 1]], axis=0)


# ======================================================================================
# Draft body (one block at a time)
# ======================================================================================


def block_forward(cfg, top, layers, emb: np.ndarray, anchor: int, slot_valid, mask_row,
                  ctx_kv, positions=None) -> np.ndarray:
    """Hidden states of one draft block ("DFlash Draft Body", How It Works step 3).

    emb [S, D] fp64: caller-supplied embeddings of the block's slots.
    anchor: the block's anchor position; slot j sits at position anchor + j (R1) unless
      `positions` [S] is given.
    slot_valid [S]: block_valid for this block (R5).
    mask_row [L]: the row's input mask (context keys need mask = 1).
    ctx_kv: per layer (K [Hkv, Lc, dh], V [Hkv, Lc, dh]) for context positions 0..Lc-1,
      Lc >= min(anchor, L).

    R6 key set for every valid query of the block: context positions c < anchor with
    mask[c] = 1 (the strict prefix: "a predicted block must not read target features
    containing its future answers", "DFlash: drafting, verification, and speed", One
    DFlash generation cycle) and every valid slot of the same block (the block is updated
    together; never another block).  Softmax(q.k / sqrt(dh)); GQA: query head h reads KV
    head h // (Hq / Hkv).
    R9 layer: pre-norm; x += W_o Attn(RMSNorm(x; g_in));
    x += W_down(SiLU(h W_gate^T) * (h W_up^T)), h = RMSNorm(x; g_post);
    output RMSNorm(x; g_final) when cfg.final_norm; exactly 0 at invalid slots."""
    S, D = emb.shape
    Hq, Hkv, dh = cfg.num_heads, cfg.num_kv_heads, cfg.head_dim
    grp = Hq // Hkv
    I = cfg.intermediate
    slot_valid = np.asarray(slot_valid).astype(bool)
    out = np.zeros((S, D), np.float64)
    if anchor < 0 or not slot_valid.any():
        return out
    pos = anchor + np.arange(S) if positions is None else np.asarray(positions)
    L = len(mask_row)
    ctx_idx = np.array([c for c in range(min(anchor, L)) if mask_row[c] != 0], dtype=np.int64)
    blk_idx = np.nonzero(slot_valid)[0]
    x = emb.astype(np.float64).copy()
    scale = 1.0 / math.sqrt(dh)
    qw, kw = Hq * dh, Hkv * dh
    for l in range(cfg.num_layers):
        lw = layers(l)
        h = rms_norm(x, lw["g_in"], cfg.rms_eps)
        qkv = h @ lw["w_qkv"].T
        q = apply_rope(qkv[:, :qw].reshape(S, Hq, dh), pos, cfg.rope_theta)
        k = apply_rope(qkv[:, qw:qw + kw].reshape(S, Hkv, dh), pos, cfg.rope_theta)
        v = qkv[:, qw + kw:].reshape(S, Hkv, dh)
        kc, vc = ctx_kv[l]
        attn = np.zeros((S, Hq, dh), np.float64)
        for hq in range(Hq):
            g = hq // grp
            keys = np.concatenate([kc[g][ctx_idx], k[blk_idx, g]], axis=0)
            vals = np.concatenate([vc[g][ctx_idx], v[blk_idx, g]], axis=0)
            p = softmax_rows((q[blk_idx, hq] @ keys.T) * scale)
            attn[blk_idx, hq] = p @ vals
        x = x + attn.reshape(S, qw) @ lw["w_o"].T
        h2 = rms_norm(x, lw["g_post"], cfg.rms_eps)
        gu = h2 @ lw["w_gate_up"].T
        x = x + (silu(gu[:, :I]) * gu[:, I:]) @ lw["w_down"].T
    y = rms_norm(x, top["g_final"], cfg.rms_eps) if cfg.final_norm else x
    out[slot_valid] = y[slot_valid]
    return out


def body_forward(cfg, top, layers, emb, anchors, block_valid, mask, ctx_kv_rows,
                 position_ids=None) -> np.ndarray:
    """All blocks: emb [B, N, S, D]; anchors [B, N]; block_valid [B, N, S]; mask [B, L];
    ctx_kv_rows: b -> per-layer context K/V of row b.  Returns [B, N, S, D] fp64."""
    B, N, S, D = emb.shape
    out = np.zeros((B, N, S, D), np.float64)
    for b in range(B):
        kv = None
        for k in range(N):
            a = int(anchors[b, k])
            if a < 0 or not np.any(block_valid[b, k]):
                continue
            if kv is None:
                kv = ctx_kv_rows(b)
            pos = None if position_ids is None else position_ids[b, k]
            out[b, k] = block_forward(cfg, top, layers, emb[b, k], a, block_valid[b, k],
                                      mask[b], kv, pos)
    return out


# ======================================================================================
# Greedy verification
# ======================================================================================


def argmax_lowest(row: np.ndarray) -> int:
    """R10: index of the largest value; ties go to the lowest index.  Values are compared
    exactly (bf16/fp32 inputs widen to fp64 without rounding)."""
    best_i, best_v = 0, row[0]
    for i in range(1, len(row)):
        if row[i] > best_v:
            best_i, best_v = i, row[i]
    return best_i


def argmax_lowest_fast(rows: np.ndarray) -> np.ndarray:
    """argmax_lowest over the last axis, vectorised (np.argmax returns the first
    occurrence of the maximum).  Pinned to argmax_lowest by the tests."""
    return np.argmax(rows, axis=-1)


def verify_greedy_block(draft, target_choices, eos_token=None):
    """Greedy block verification ("DFlash: drafting, verification, and speed", One DFlash
    generation cycle): accept the longest prefix of the draft that agrees with the
    target's choices; at the first disagreement emit the target's own choice and stop;
    if every proposal agrees, also emit the last target choice (the bonus); a matched
    EOS proposal ends the block at once (no bonus).  target_choices must hold one entry
    per draft token plus the bonus, else ValueError.  Returns (emitted, accepted)."""
    draft, choices = list(draft), list(target_choices)
    if len(choices) != len(draft) + 1:
        raise ValueError("target_choices needs len(draft) + 1 entries")
    n = 0
    while n < len(draft) and draft[n] == choices[n]:
        n += 1
        if eos_token is not None and draft[n - 1] == eos_token:
            return draft[:n], n
    if n == len(draft):
        return draft + [choices[-1]], n
    return draft[:n] + [choices[n]], n


def verify_greedy(logits: np.ndarray, draft: np.ndarray, eos: int = -1):
    """Batched greedy verification.  logits [B, gamma+1, V] (R11: row i is the target's
    distribution after the anchor and draft[0..i-1]); draft [B, gamma]; eos < 0 = none.
    Returns (choices [B, gamma+1], emitted [B, gamma+1] padded with -1,
    num_emitted [B], accepted [B]), all int32."""
    B, S, V = logits.shape
    if draft.shape != (B, S - 1):
        raise ValueError("draft must be [B, gamma] with gamma + 1 logits rows per request")
    choices = argmax_lowest_fast(logits).astype(np.int32)
    emitted = np.full((B, S), -1, np.int32)
    num = np.zeros(B, np.int32)
    acc = np.zeros(B, np.int32)
    for b in range(B):
        e, a = verify_greedy_block([int(t) for t in draft[b]], [int(c) for c in choices[b]],
                                   None if eos < 0 else eos)
        emitted[b, :len(e)] = e
        num[b] = len(e)
        acc[b] = a
    return choices, emitted, num, acc


# ======================================================================================
# Speculative-sampling verification
# ======================================================================================


def counter_uniform(seed: int, *counters: int) -> float:
    """Counter-based uniform draw in (0, 1): the SplitMix64 finaliser chained over the seed
    and the counters (each taken as uint64), as anchor_key chains it; the top 23 bits of
    the result plus one half, times 2^-23.  Every value is an odd multiple of 2^-24 strictly
    inside (0, 1) with at most 24 significant bits, exact in fp32 and fp64, so both sides of
    a comparison draw identical numbers from identical counters."""
    h = splitmix64_mix(seed & U64)
    for c in counters:
        h = splitmix64_mix(h ^ (c & U64))
    return ((h >> 41) + 0.5) * 2.0 ** -23


def race_sample(weights: np.ndarray, seed: int, *counters: int) -> int:
    """One draw from weights / sum(weights) (weights >= 0, at least one > 0) by the
    exponential race: every index v with w_v > 0 gets an arrival time E_v / w_v with E_v =
    -ln U_v i.i.d. Exp(1) (U_v = counter_uniform(seed, *counters, v)); the first arrival
    wins (lowest index on an exact tie).  The minimum of independent exponentials of rates
    w_v is attained at v with probability w_v / sum(w), so the draw is exact and needs no
    normalisation or cumulative sum."""
    best, best_t = -1, math.inf
    for v in range(len(weights)):
        w = float(weights[v])
        if w > 0.0:
            t = -math.log(counter_uniform(seed, *counters, v)) / w
            if t < best_t:
                best, best_t = v, t
    return best


def verify_sampling_block(p_rows: np.ndarray, q_rows: np.ndarray, draft, seed: int, b: int,
                          eos_token=None):
    """Speculative-sampling verification of one drafted block ("DFlash: drafting,
    verification, and speed", Sampling with temperature is not argmax matching).

    p_rows [gamma+1, V]: the target's distributions (row i after the anchor and draft[:i]);
    q_rows [gamma, V]: the ACTUAL proposal distributions the draft tokens were drawn from
    (after any top-k, temperature or selector).  For each proposal y = draft[i] in order:
    accept with probability min(1, p_i(y) / q_i(y)) -- drawn as U < p_i(y) / q_i(y) with
    U = counter_uniform(seed, b, i, 0); on the first rejection emit a sample of the
    normalised residual [p_i - q_i]_+ and stop.  When every proposal is accepted, the block
    ends with a sample of p_gamma, the counterpart of greedy verification's bonus token (this
    reading: the pages state the acceptance and residual rules only).  A matched EOS
    proposal ends the block as in greedy verification.  Samples use race_sample with
    counters (b, i, 1).  If the residual is zero everywhere (p_i == q_i, where a rejection
    cannot happen in exact arithmetic) the sample is drawn from p_i.
    Returns (emitted, accepted)."""
    draft = [int(t) for t in draft]
    gamma = len(draft)
    if p_rows.shape[0] != gamma + 1 or q_rows.shape[0] != gamma:
        raise ValueError("need gamma + 1 target rows and gamma proposal rows")
    out, acc = [], 0
    for i, y in enumerate(draft):
        u = counter_uniform(seed, b, i, 0)
        py, qy = float(p_rows[i, y]), float(q_rows[i, y])
        if u * qy < py:            # U < p/q, with q(y) = 0 always accepted
            out.append(y)
            acc += 1
            if eos_token is not None and y == eos_token:
                return out, acc
            continue
        r = np.maximum(p_rows[i] - q_rows[i], 0.0)
        out.append(race_sample(r if np.any(r > 0) else p_rows[i], seed, b, i, 1))
        return out, acc
    out.append(race_sample(p_rows[gamma], seed, b, gamma, 1))
    return out, acc


def verify_sampling(logits: np.ndarray, temperature: float, q: np.ndarray, draft: np.ndarray,
                    seed: int, eos: int = -1):
    """Batched speculative-sampling verification.  logits [B, gamma+1, V] (the target's
    distribution p = softmax(logits / temperature) per row, temperature > 0), q [B, gamma, V]
    the actual proposal distributions, draft [B, gamma].  Returns (emitted [B, gamma+1]
    padded with -1, num_emitted [B], accepted [B]), int32."""
    B, S, V = logits.shape
    if draft.shape != (B, S - 1) or q.shape != (B, S - 1, V) or not temperature > 0:
        raise ValueError("need draft [B, gamma], q [B, gamma, V] and temperature > 0")
    emitted = np.full((B, S), -1, np.int32)
    num = np.zeros(B, np.int32)
    acc = np.zeros(B, np.int32)
    for b in range(B):
        p = softmax_rows(np.asarray(logits[b], np.float64) / temperature)
        e, a = verify_sampling_block(p, np.asarray(q[b], np.float64), draft[b], seed, b,
                                     None if eos < 0 else eos)
        emitted[b, :len(e)] = e
        num[b] = len(e)
        acc[b] = a
    return emitted, num, acc


# ======================================================================================
# Training loss over the drafted blocks
# ======================================================================================


def position_weights(block_size: int, decay: float) -> np.ndarray:
    """Loss weight of each block slot.  "DFlash" (How it works, Loss): cross-entropy with an
    exponential positional decay that weights earlier in-block positions more heavily;
    "DFlash: drafting, verification, and speed" (One DFlash generation cycle): greater loss
    weight on early positions.  The pages give no constant.  Reading: slot j >= 1 (the
    first predicted position is j = 1) weighs exp(-(j - 1) / decay), decay > 0 a caller
    argument; the anchor slot j = 0 weighs 0 (loss_mask excludes it anyway)."""
    if not decay > 0:
        raise ValueError("decay must be > 0")
    w = np.zeros(block_size, np.float64)
    j = np.arange(1, block_size, dtype=np.float64)
    w[1:] = np.exp(-(j - 1.0) / decay)
    return w


def decayed_ce_loss(hidden: np.ndarray, w_lm: np.ndarray, targets: np.ndarray,
                    loss_mask: np.ndarray, decay: float):
    """Draft loss of a batch of blocks: per slot, the cross-entropy of the frozen lm_head's
    logits (hidden W_lm^T) against the ground-truth token, weighted by position_weights and
    by loss_mask ("DFlash Draft Body", How It Works step 4: the loss mask excludes the anchor
    and invalid positions); loss = sum(m w CE) / sum(m w) (0 when nothing is weighted).

    hidden [B, N, S, D] (the body's output), w_lm [V, D], targets [B, N, S] int (read where
    loss_mask is set), loss_mask [B, N, S].  Returns (loss, ce [B, N, S] with 0 where the
    mask is 0)."""
    B, N, S, D = hidden.shape
    w = position_weights(S, decay)
    ce = np.zeros((B, N, S), np.float64)
    idx = np.argwhere(np.asarray(loss_mask) != 0)          # masked slots (b, k, j)
    if len(idx) == 0:
        return 0.0, ce
    logits = hidden[idx[:, 0], idx[:, 1], idx[:, 2]] @ w_lm.T   # [slots, V], one matmul
    num = den = 0.0
    for r, (b, k, j) in enumerate(idx):
        m = np.max(logits[r])
        lse = m + math.log(np.sum(np.exp(logits[r] - m)))
        ce[b, k, j] = lse - logits[r, int(targets[b, k, j])]
        num += w[j] * ce[b, k, j]
        den += w[j]
    return (num / den if den > 0 else 0.0), ce

