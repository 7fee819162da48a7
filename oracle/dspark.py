"""Plain, slow, fp64 CPU statement of one DSpark draft-head round.

TEST INFRASTRUCTURE.  This oracle exists to check the CUDA path.  Only tests/,
__graft_entry__.smoke() and bench.py's CPU-baseline leg may import or call it;
the product path never does, and it shares no code with the CUDA library.

Pages followed (by title and section):
  [DD]  "大模型推理的'免费加速'还能怎么卷？DSpark 深度解读" (zhichai.net)
        §二 设计一: Markov head  B(x_{k-1},.) = W1[x_{k-1}] W2, W1: V x r, W2: r x V
        §二 设计二: confidence head c_k = sigmoid(w^T [h_k; W1[x_{k-1}]]),
              label c* = 1 - 1/2 ||p_d - p_t||_1, Sequential Temperature Scaling,
              hardware-aware prefix scheduler Theta = tau * SPS(B),
              B = sum(1 + l_r), tau = sum(1 + sum_j a_{r,j}), a_{r,j} = prod_i c_{r,i},
              global descending sort, greedy admission with a break
        §三 挑战1/挑战2: asynchronous top-K, unconstrained search without the break
  [AR]  "DSpark整体架构" (10100.com), Fig. 1 and the semi-autoregressive stages:
        the anchor is itself the first prediction position; verification keeps
        the accepted run and emits one corrected token.
  [V4]  DeepSeek-V4-Pro-0813 DSpark article (demingchina.com), config table:
        block size 5, markov rank 512, noise token 128799, fp32 confidence.

Readings where the pages are silent (each listed in the design notes):
  * x_0 = anchor: bias and confidence at position 1 use the anchor's W1 row.
  * T_k divides the confidence logit: c_k = sigmoid(z_k / T_k).  No bias term.
  * Sampling temperature tau divides (base + bias); tau = 0 means greedy argmax
    (ties to the lowest vocabulary id); tau > 0 samples by Gumbel-max with the
    Philox layout of oracle.philox, in two levels over blocks of 64 vocabulary
    entries (gumbel_max below).  The target uses the same tau.
  * Base logits are materialised in bf16 (the LM head's output type); every
    later step accumulates in float64 here.
  * Confidences are float32; survival products a_{r,j} are float32 products
    taken left to right (the scheduler's sort is decided in that precision);
    S_K is the exact sum of the sorted products each rounded to the nearest
    multiple of 2^-48, and Theta(K) = f64(R + S_K) * (f64(SPS) * 2^-48), so
    the argmax over K is decided in the same precision as on the device.
    The rounding moves R + S_K by at most gamma * 2^-49 of itself.
  * Sort order: a descending, ties by (request, position) ascending.
    Theta argmax ties go to the smallest K; the break mode admits K+1 only if
    Theta(K+1) > Theta(K) strictly.
  * Verification is standard speculative sampling: accept x_j iff
    u * p_d(x_j) < p_t(x_j); on the first rejection sample from
    norm(max(0, p_t - p_d)); if every draft is accepted, sample the bonus from
    target row l_r + 1.  Greedy: accept iff x_j = argmax t_j.
  * The residual draw is by rejection from p_t: trial q proposes y ~ p_t and
    keeps it iff u_q p_t(y) < p_t(y) - p_d(y), so a kept y has law
    max(0, p_t - p_d) / sum(max(0, p_t - p_d)) exactly (von Neumann's
    rejection method with envelope p_t, whose ratio max(0, p_t - p_d) / p_t is
    at most 1).  The first kept of RESIDUAL_TRIALS trials is the token; when
    none is kept, the residual is formed explicitly and drawn by Gumbel-max.
    A proposal is a three-level Gumbel-max draw (gumbel_max_trial): over
    super-blocks of 16 sampler blocks (1024 ids), over the sampler blocks of
    the winning super-block, then over the ids of the winning block, so a
    trial needs a few hundred random words rather than one per block.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np

from . import philox

UNCONSTRAINED = 0
BREAK = 1
FIXED_K = 2


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def to_f64(x) -> np.ndarray:
    """Accept numpy arrays or torch tensors (any float dtype) and return float64."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        if str(x.dtype) == "torch.bfloat16":
            x = x.float()
        x = x.numpy()
    return np.asarray(x, dtype=np.float64)


def to_i64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.asarray(x, dtype=np.int64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round to bfloat16 (via float32, round-to-nearest-even), returned in float64."""
    f = np.asarray(x, dtype=np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) & np.uint64(0xFFFF0000)
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def logsumexp(x: np.ndarray, axis: int = -1) -> np.ndarray:
    m = np.max(x, axis=axis, keepdims=True)
    return (m + np.log(np.sum(np.exp(x - m), axis=axis, keepdims=True))).squeeze(axis)


def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def top2_margin(score: np.ndarray) -> np.ndarray:
    """Difference between the largest and second-largest entry of each row."""
    part = np.partition(score, -2, axis=-1)
    return part[..., -1] - part[..., -2]


def _block_logsumexp(x: np.ndarray) -> np.ndarray:
    """logsumexp over the last axis; -inf for an all -inf row (an empty block)."""
    m = np.max(x, axis=-1, keepdims=True)
    finite = np.isfinite(m)
    safe = np.where(finite, m, 0.0)
    with np.errstate(divide="ignore"):
        out = safe + np.log(np.sum(np.exp(x - safe), axis=-1, keepdims=True))
    return np.where(finite, out, -np.inf).squeeze(-1)


# ---------------------------------------------------------------------------
# the sampler shared by every random draw of the round
# ---------------------------------------------------------------------------

GUMBEL_BLOCK = 64
RESIDUAL_TRIALS = 64   # proposals from p_t per rejected row before the explicit residual
TRIAL_SUPER = 16       # sampler blocks per first-level block of a trial proposal


def gumbel_max(score, seed: int, position, request, stream: int,
               block: int = GUMBEL_BLOCK) -> Dict[str, np.ndarray]:
    """One draw from softmax(score) per row, by Gumbel-max in two levels.

    score [N, V] float64 log-weights (-inf excludes an entry); position and
    request broadcast to [N].  The pages name Gumbel-max keyed by
    (seed, request, position) and fix nothing further; this is the reading:

      1. cut the vocabulary into blocks of `block` consecutive ids (the last
         one shorter when V is not a multiple);
      2. block b scores G_b = log sum_{v in b} e^{score_v} + g_b, g_b the Gumbel
         of block id b in stream `stream + 4`;
      3. b* = argmax_b G_b (lowest b on ties; blocks of zero mass never win);
      4. the token is argmax over v in b* of score_v + g_v, g_v the Gumbel of
         vocabulary id v in stream `stream` (lowest v on ties).

    Exactness (max-stability of the Gumbel law): max_{v in b}(score_v + g_v)
    is Gumbel with location log Z_b, so step 3 picks b with probability
    Z_b / Z and step 4 picks v in b with probability e^{score_v} / Z_b; the
    product is softmax(score)_v (Maddison, Tarlow, Minka, "A* Sampling",
    NIPS 2014, on the top-down construction of Gumbel processes).

    Returns token [N] (-1 when every entry is -inf), margin [N] (the smaller
    of the two levels' top-2 gaps; +inf where a level has one candidate),
    block_scores [N, nb] and entry_scores [N, V] (score + g for every id).
    """
    score = np.atleast_2d(to_f64(score))
    N, V = score.shape
    nb = (V + block - 1) // block
    pos = np.broadcast_to(np.asarray(position, dtype=np.uint64), (N,))
    req = np.broadcast_to(np.asarray(request, dtype=np.uint64), (N,))
    padded = np.full((N, nb * block), -np.inf)
    padded[:, :V] = score
    lse_b = _block_logsumexp(padded.reshape(N, nb, block))
    g_b = philox.gumbel(seed, pos[:, None], req[:, None], stream + philox.BLOCK_STREAM_OFFSET,
                        np.arange(nb, dtype=np.uint64)[None, :])
    G = lse_b + g_b                                      # -inf for empty blocks
    g_v = philox.gumbel(seed, pos[:, None], req[:, None], stream,
                        np.arange(V, dtype=np.uint64)[None, :])
    e = score + g_v
    bstar = np.argmax(G, axis=1)
    token = np.full(N, -1, dtype=np.int64)
    margin = np.full(N, np.inf)
    for n in range(N):
        if not np.isfinite(G[n, bstar[n]]):
            continue
        lo, hi = bstar[n] * block, min(V, bstar[n] * block + block)
        inner = e[n, lo:hi]
        token[n] = lo + int(np.argmax(inner))
        gb = G[n][np.isfinite(G[n])]
        gi = inner[np.isfinite(inner)]
        m_b = top2_margin(gb) if gb.size > 1 else np.inf
        m_i = top2_margin(gi) if gi.size > 1 else np.inf
        margin[n] = min(m_b, m_i)
    return dict(token=token, margin=margin, block_scores=G, entry_scores=e)


def gumbel_max_trial(score, seed: int, position: int, request: int, stream: int,
                     block: int = GUMBEL_BLOCK, sup: int = TRIAL_SUPER) -> Dict[str, float]:
    """One draw from softmax(score) (score [V] float64 log-weights) in three levels:

      1. super-blocks of sup * block consecutive ids: S* = argmax_S log Z_S + g_S,
         g_S the Gumbel of super-block id S in stream `stream + 5`;
      2. blocks of `block` ids inside S*: b* = argmax_b log Z_b + g_b, g_b the
         Gumbel of block id b (numbered over the whole vocabulary) in stream
         `stream + 4`;
      3. ids inside b*: argmax_v score_v + g_v, g_v the Gumbel of id v in stream
         `stream`.
    Lowest index on ties; parts of zero mass never win.  Max-stability makes
    each level pick its part with probability proportional to its mass given the
    level above, so the token has probability softmax(score)_v (the top-down
    construction of gumbel_max, one level deeper).  Returns token (-1 when every
    entry is -inf) and margin (the smallest of the three levels' top-2 gaps).
    """
    score = to_f64(score).reshape(-1)
    V = score.size
    nb = (V + block - 1) // block
    ns = (nb + sup - 1) // sup
    padded = np.full(ns * sup * block, -np.inf)
    padded[:V] = score
    lz_b = _block_logsumexp(padded.reshape(ns * sup, block))          # [ns * sup]
    lz_s = _block_logsumexp(lz_b.reshape(ns, sup))                     # [ns]
    out = dict(token=-1, margin=np.inf)

    def pick(vals, ids, st):
        g = philox.gumbel(seed, position, request, st, np.asarray(ids, dtype=np.uint64))
        e = vals + g
        fin = np.isfinite(vals)
        if not np.any(fin):
            return -1, np.inf
        k = int(np.argmax(np.where(fin, e, -np.inf)))
        ef = e[fin]
        return int(ids[k]), (top2_margin(ef) if ef.size > 1 else np.inf)

    S, m1 = pick(lz_s, np.arange(ns), stream + 5)
    if S < 0:
        return out
    bs = np.arange(S * sup, min(nb, S * sup + sup))
    b, m2 = pick(lz_b[bs], bs, stream + 4)
    vs = np.arange(b * block, min(V, b * block + block))
    v, m3 = pick(score[vs], vs, stream)
    out["token"] = v
    out["margin"] = min(m1, m2, m3)
    return out


# ---------------------------------------------------------------------------
# a1: base logits through the shared, frozen LM head   [DD §二 architecture; AR]
# ---------------------------------------------------------------------------

def base_logits(h, W_lm, bf16_out: bool = True, vocab_chunk: int = 0) -> np.ndarray:
    """l0[m, v] = sum_i h[m, i] W_lm[v, i]  (W_lm stored [V, d]).

    h is [..., d]; the result is [..., V].  `vocab_chunk` > 0 only splits the
    vocabulary into slices to bound host memory; each slice is the same matmul.
    """
    h = to_f64(h)
    lead = h.shape[:-1]
    h2 = h.reshape(-1, h.shape[-1])
    if vocab_chunk and vocab_chunk < W_lm.shape[0]:
        parts = []
        for v0 in range(0, W_lm.shape[0], vocab_chunk):
            parts.append(h2 @ to_f64(W_lm[v0:v0 + vocab_chunk]).T)
        out = np.concatenate(parts, axis=1)
    else:
        out = h2 @ to_f64(W_lm).T
    if bf16_out:
        out = round_bf16(out)
    return out.reshape(*lead, -1)


# ---------------------------------------------------------------------------
# a2-a4: gamma-step Markov-head loop with the confidence head
#        [DD §二 设计一 and 设计二 confidence head; AR semi-autoregressive stage 2]
# ---------------------------------------------------------------------------

def markov_draft(base, h, anchor, W1, W2, w_conf, T, tau: float, seed: int,
                 forced=None, keep_logits: bool = False, keep_scores: bool = False,
                 requests: Optional[np.ndarray] = None,
                 block: int = GUMBEL_BLOCK) -> Dict[str, np.ndarray]:
    """Run the sequential head for k = 1..gamma.

    base [R, gamma, V] base logits; h [R, gamma, d]; anchor [R]; W1 [V, r];
    W2 [r, V]; w_conf [d + r]; T [gamma]; tau sampling temperature (0 = greedy).
    `forced` [R, gamma]: when given, step k conditions on forced[:, k-1] instead
    of the oracle's own x_k (used to evaluate the draft distribution along a
    given token path, e.g. for verification).  `requests` gives the request ids
    used for the random streams (default 0..R-1).  `keep_scores` returns the
    decision score of every vocabulary entry at every step (sampling: also the
    block scores of gumbel_max).  `block` is the sampler's block width.

    Returns tokens (the oracle's own choice at each step), conf, z, margin (top-2
    gap of the decision score), and in sampling mode lse = logsumexp(l_k / tau)
    and logp = l_k[x_k] / tau - lse for the token that conditions the next step.
    """
    base = to_f64(base)
    h = to_f64(h)
    anchor = to_i64(anchor)
    W1 = to_f64(W1)
    W2 = to_f64(W2)
    w_conf = to_f64(w_conf)
    T = to_f64(T)
    R, G, V = base.shape
    d = h.shape[-1]
    w_h, w_e = w_conf[:d], w_conf[d:]
    req = np.arange(R) if requests is None else to_i64(requests)

    tokens = np.zeros((R, G), dtype=np.int64)
    conf = np.zeros((R, G))
    z_out = np.zeros((R, G))
    margin = np.zeros((R, G))
    lse = np.zeros((R, G))
    logp = np.zeros((R, G))
    path = np.zeros((R, G), dtype=np.int64)
    logits = np.zeros((R, G, V)) if keep_logits else None
    scores = np.zeros((R, G, V)) if keep_scores else None
    nb = (V + block - 1) // block
    bscores = np.zeros((R, G, nb)) if keep_scores and tau != 0.0 else None
    forced = None if forced is None else to_i64(forced)

    prev = anchor.copy()
    for k in range(1, G + 1):
        e = W1[prev]                                   # [R, r]  W1[x_{k-1}]
        ell = base[:, k - 1, :] + e @ W2               # base + B(x_{k-1}, .)
        z = h[:, k - 1, :] @ w_h + e @ w_e             # w^T [h_k; W1[x_{k-1}]]
        conf[:, k - 1] = sigmoid(z / T[k - 1])
        z_out[:, k - 1] = z
        if tau == 0.0:
            score = ell
            x = np.argmax(score, axis=1)               # first maximum: lowest id
            margin[:, k - 1] = top2_margin(score)
        else:
            smp = gumbel_max(ell / tau, seed, k, req, philox.STREAM_DRAFT, block)
            score = smp["entry_scores"]
            x = smp["token"]
            margin[:, k - 1] = smp["margin"]
            if bscores is not None:
                bscores[:, k - 1, :] = smp["block_scores"]
        tokens[:, k - 1] = x
        nxt = x if forced is None else forced[:, k - 1]
        path[:, k - 1] = nxt
        if tau != 0.0:
            lse[:, k - 1] = logsumexp(ell / tau, axis=1)
            logp[:, k - 1] = ell[np.arange(R), nxt] / tau - lse[:, k - 1]
        if keep_logits:
            logits[:, k - 1, :] = ell
        if keep_scores:
            scores[:, k - 1, :] = score
        prev = nxt
    out = dict(tokens=tokens, conf=conf, z=z_out, margin=margin, lse=lse, logp=logp,
               path=path)
    if keep_logits:
        out["logits"] = logits
    if keep_scores:
        out["scores"] = scores
        if bscores is not None:
            out["block_scores"] = bscores
            out["block"] = block
    return out


# ---------------------------------------------------------------------------
# a1 + a2 fused: one contraction per step   [DD §二 设计一]
# ---------------------------------------------------------------------------


def fused_draft(h, anchor, W_lm, W1, W2, w_conf, T, tau: float, seed: int,
                **kw) -> Dict[str, np.ndarray]:
    """The same draft head with the base logits never materialised.

    One contraction per step, [h_k; W1[x_{k-1}]] . [W_lm; W2]^T, gives the whole
    draft logit, so h_k . W_lm is not rounded to bf16 as the LM head's stored
    output is; everything else is markov_draft's."""
    return markov_draft(base_logits(h, W_lm, bf16_out=False), h, anchor, W1, W2, w_conf, T,
                        tau, seed, **kw)


# ---------------------------------------------------------------------------
# a2': the RNN head variant   [AR stage two, "RNN head"; DD §二 设计一]
# ---------------------------------------------------------------------------


def rnn_draft(base, h, anchor, W1, W2, W_gc, w_conf, T, tau: float, seed: int,
              keep_scores: bool = False, block: int = GUMBEL_BLOCK) -> Dict[str, np.ndarray]:
    """The sequential head with a gated in-block recurrent state.

    The pages describe it only in words: a block-internal recurrent state,
    updated by a gated step over the concatenation of the history (the state),
    the previous token's embedding and the backbone hidden state.  Reading:
      u_k  = [s_{k-1}; W1[x_{k-1}]; h_k]          (s_0 = 0, x_0 = anchor)
      g_k  = sigmoid(W_g u_k),  c_k~ = tanh(W_c u_k),   W_gc = [W_g; W_c]  [2r, 2r + d]
      s_k  = (1 - g_k) * s_{k-1} + g_k * c_k~
      l_k  = base_k + s_k W2                      (the Markov head's low-rank output map)
    The state enters each contraction rounded to bf16 (an activation, like the
    base logits); it is carried in float64 between steps.  Sampling, the
    confidence head (on [h_k; W1[x_{k-1}]]) and the outputs are markov_draft's.
    """
    base = to_f64(base)
    h = to_f64(h)
    anchor = to_i64(anchor)
    W1 = to_f64(W1)
    W2 = to_f64(W2)
    W_gc = to_f64(W_gc)
    w_conf = to_f64(w_conf)
    T = to_f64(T)
    R, G, V = base.shape
    d = h.shape[-1]
    r = W1.shape[1]
    w_h, w_e = w_conf[:d], w_conf[d:]
    req = np.arange(R)
    tokens = np.zeros((R, G), dtype=np.int64)
    conf = np.zeros((R, G))
    margin = np.zeros((R, G))
    lse = np.zeros((R, G))
    logp = np.zeros((R, G))
    scores = np.zeros((R, G, V)) if keep_scores else None
    nb = (V + block - 1) // block
    bscores = np.zeros((R, G, nb)) if keep_scores and tau != 0.0 else None
    state = np.zeros((R, r))
    prev = anchor.copy()
    for k in range(1, G + 1):
        e = W1[prev]                                              # W1[x_{k-1}]
        u = np.concatenate([round_bf16(state), e, h[:, k - 1, :]], axis=1)
        pre = u @ W_gc.T                                          # [R, 2r]
        g = sigmoid(pre[:, :r])
        cand = np.tanh(pre[:, r:])
        state = (1.0 - g) * state + g * cand
        ell = base[:, k - 1, :] + round_bf16(state) @ W2
        z = h[:, k - 1, :] @ w_h + e @ w_e
        conf[:, k - 1] = sigmoid(z / T[k - 1])
        if tau == 0.0:
            score = ell
            x = np.argmax(score, axis=1)
            margin[:, k - 1] = top2_margin(score)
        else:
            smp = gumbel_max(ell / tau, seed, k, req, philox.STREAM_DRAFT, block)
            score = smp["entry_scores"]
            x = smp["token"]
            margin[:, k - 1] = smp["margin"]
            if bscores is not None:
                bscores[:, k - 1, :] = smp["block_scores"]
            lse[:, k - 1] = logsumexp(ell / tau, axis=1)
            logp[:, k - 1] = ell[np.arange(R), x] / tau - lse[:, k - 1]
        tokens[:, k - 1] = x
        if keep_scores:
            scores[:, k - 1, :] = score
        prev = x
    out = dict(tokens=tokens, conf=conf, margin=margin, lse=lse, logp=logp, state=state)
    if keep_scores:
        out["scores"] = scores
        if bscores is not None:
            out["block_scores"] = bscores
            out["block"] = block
    return out


# ---------------------------------------------------------------------------
# a5-a7: survival products, global sort, Theta search   [DD §二 scheduler, §三]
# ---------------------------------------------------------------------------

def survival(conf) -> np.ndarray:
    """a_{r,j} = prod_{i<=j} c_{r,i}, float32 products taken left to right."""
    c = np.asarray(to_f64(conf), dtype=np.float32)
    a = np.empty_like(c)
    a[:, 0] = c[:, 0]
    for j in range(1, c.shape[1]):
        a[:, j] = a[:, j - 1] * c[:, j]
    return a


def global_order(a: np.ndarray) -> np.ndarray:
    """Flat candidate ids r*gamma + (j-1), sorted by a descending, ties by id ascending."""
    flat = a.reshape(-1)
    return np.array(sorted(range(flat.size), key=lambda i: (-float(flat[i]), i)),
                    dtype=np.int64)


FIX_BITS = 48  # S_K is summed in units of 2^-48


def theta_curve(a: np.ndarray, order: np.ndarray, sps) -> np.ndarray:
    """Theta(K) = (R + S_K) * SPS(R + K), K = 0..R*gamma, S_K = sum of the top-K a.

    Each a (float32 in [0, 1]) is rounded to the nearest integer number of
    2^-48 units, halves up: a * 2^48 is exact in float64 and so is adding 0.5
    (for a * 2^48 below 2^-29 the sum rounds, but stays below 1).  The sums are
    exact Python integers; R + S_K is converted to float64 once (nearest) and
    multiplied by SPS * 2^-48 (exact scaling)."""
    R = a.shape[0]
    sps = to_f64(sps)
    sorted_a = a.reshape(-1)[order].astype(np.float64)
    units = np.floor(sorted_a * 2.0 ** FIX_BITS + 0.5)
    RS = R << FIX_BITS
    theta = np.empty(units.size + 1)
    theta[0] = float(RS) * (sps[R - 1] * 2.0 ** -FIX_BITS)
    for K in range(1, units.size + 1):
        RS += int(units[K - 1])
        theta[K] = float(RS) * (sps[R + K - 1] * 2.0 ** -FIX_BITS)
    return theta


def schedule(conf, sps, mode: int = UNCONSTRAINED, k_fixed: int = 0) -> Dict[str, np.ndarray]:
    """Per-request verify lengths l_r from the confidences.

    mode UNCONSTRAINED: K = argmax_K Theta(K) over all budgets (ties: smallest K)
    mode BREAK:         admit in sorted order while Theta strictly increases
    mode FIXED_K:       admit the top min(k_fixed, R*gamma) candidates
    """
    a = survival(conf)
    R, G = a.shape
    sps = to_f64(sps)
    if sps.size < R * (G + 1):
        raise ValueError("SPS table shorter than R * (gamma + 1)")
    order = global_order(a)
    th = theta_curve(a, order, sps)
    n = R * G
    if mode == UNCONSTRAINED:
        K = int(np.argmax(np.where(np.isnan(th), -np.inf, th)))  # a NaN entry never wins
    elif mode == BREAK:
        K = 0
        while K < n and th[K + 1] > th[K]:
            K += 1
    elif mode == FIXED_K:
        K = min(max(int(k_fixed), 0), n)
    else:
        raise ValueError(mode)
    lens = np.bincount(order[:K] // G, minlength=R).astype(np.int64)
    return dict(len=lens, K=K, theta=float(th[K]), thetas=th, a=a, order=order)


def schedule_async(conf_rounds, sps, k_round0: int, k_round1: int) -> Dict[str, np.ndarray]:
    """Asynchronous admission over consecutive rounds  [DD §三 挑战1].

    Round t-2 produces confidences and predicts round t's capacity: the
    unconstrained optimum K*_{t-2} = argmax_K Theta(K) of its own candidates.
    Round t sorts its candidates by their actual survival products and admits
    the top K*_{t-2} (rounds 0 and 1 admit k_round0 and k_round1).  Returns,
    per round, len [T, R], the admitted K_used [T], the prediction K_pred [T]
    it hands to round t + 2, and Theta(K_used) [T].
    """
    pending = [int(k_round0), int(k_round1)]
    lens, used, pred, theta = [], [], [], []
    for t, conf in enumerate(conf_rounds):
        k_t = pending[t % 2]                          # predicted two rounds ago
        now = schedule(conf, sps, FIXED_K, k_t)       # top-K on this round's products
        best = schedule(conf, sps, UNCONSTRAINED)     # this round's optimum, for t + 2
        pending[t % 2] = best["K"]
        lens.append(now["len"])
        used.append(now["K"])
        pred.append(best["K"])
        theta.append(now["theta"])
    return dict(len=np.array(lens), K_used=np.array(used), K_pred=np.array(pred),
                theta=np.array(theta))


# ---------------------------------------------------------------------------
# Sequential Temperature Scaling fit   [DD §二 设计二 STS 校准; DD stage summary]
# ---------------------------------------------------------------------------

def expected_calibration_error(prob, label, n_bins: int) -> float:
    """ECE with n_bins equal-width bins over [0, 1]:
    sum over bins of |B_b| / N * |mean(label in B_b) - mean(prob in B_b)|,
    i.e. sum_b |sum_{B_b} label - sum_{B_b} prob| / N.  A value of prob falls in
    bin min(floor(prob * n_bins), n_bins - 1), decided in float32."""
    p32 = np.asarray(prob, dtype=np.float32)
    b = np.minimum((p32 * np.float32(n_bins)).astype(np.int64), n_bins - 1)
    diff = np.zeros(n_bins)
    np.add.at(diff, b, np.asarray(label, dtype=np.float64) - p32.astype(np.float64))
    return float(np.sum(np.abs(diff)) / p32.size)


def sts_fit(z, accepted, T_grid, n_bins: int) -> Dict[str, np.ndarray]:
    """Per-position temperatures fitted left to right on held-out rounds.

    z [N, gamma] confidence logits w^T [h_j; W1[x_{j-1}]] (before the
    temperature); accepted [N] drafts accepted when all gamma were verified.
    Position j calibrates the prefix survival a_j = a_{j-1} * sigmoid(z_j / T)
    (float32, left to right, as the scheduler takes it) against the label
    "positions 1..j all accepted": every T of T_grid is tried with T_1..T_{j-1}
    already fixed, and the one of least ECE is kept (ties: the earliest in the
    grid).  Returns T [gamma], ece [gamma] (the ECE at the chosen T) and
    ece_grid [gamma, n_grid] (every candidate's ECE).
    """
    z32 = np.asarray(z, dtype=np.float32)
    acc = np.asarray(accepted, dtype=np.int64)
    grid = np.asarray(T_grid, dtype=np.float32)
    N, G = z32.shape
    a_prev = np.ones(N, dtype=np.float32)
    T_out = np.zeros(G, dtype=np.float32)
    ece_out = np.zeros(G)
    ece_grid = np.zeros((G, grid.size))
    for j in range(G):
        label = (acc >= j + 1).astype(np.float64)
        best_e, best_g, best_a = np.inf, 0, None
        for g, T in enumerate(grid):
            c = np.float32(1.0) / (np.float32(1.0) + np.exp(-(z32[:, j] / T)))
            a = a_prev * c if j else c
            e = expected_calibration_error(a, label, n_bins)
            ece_grid[j, g] = e
            if e < best_e:
                best_e, best_g, best_a = e, g, a
        T_out[j] = grid[best_g]
        ece_out[j] = best_e
        a_prev = best_a
    return dict(T=T_out, ece=ece_out, ece_grid=ece_grid)


def theta_of_lengths(a: np.ndarray, lens, sps) -> float:
    """Theta for an explicit allocation: B = sum(1 + l_r), tau = sum(1 + sum_{j<=l_r} a_{r,j})."""
    sps = to_f64(sps)
    lens = to_i64(lens)
    a64 = a.astype(np.float64)
    B = int(np.sum(1 + lens))
    tau = float(sum(1.0 + a64[r, :lens[r]].sum() for r in range(a.shape[0])))
    return tau * sps[B - 1]


# ---------------------------------------------------------------------------
# a8: verification   [AR Fig. 1; DD §二 losslessness; standard speculative sampling]
# ---------------------------------------------------------------------------

def confidence_label(p_d: np.ndarray, p_t: np.ndarray) -> np.ndarray:
    """c* = 1 - 1/2 ||p_d - p_t||_1 over the last axis  [DD §二 confidence label]."""
    return 1.0 - 0.5 * np.sum(np.abs(p_d - p_t), axis=-1)


def verify(tokens, lens, draft_logits, target, tau: float, seed: int,
           requests: Optional[np.ndarray] = None,
           block: int = GUMBEL_BLOCK) -> Dict[str, np.ndarray]:
    """Verify each request's admitted prefix against the target.

    tokens [R, gamma]; lens [R]; draft_logits [R, gamma, V] (final l_k, only
    read in sampling mode); target [R, gamma + 1, V] target logits, row j-1 is
    the target's distribution for draft position j.
    Returns accepted [R], bonus [R], and diagnostics: accept_margin [R, gamma]
    (log u + log p_d - log p_t at each tested position, nan elsewhere) and
    final_margin [R] (top-2 gap of the score that picked the bonus; sampling:
    the margin of gumbel_max, and for residual trials the smallest of every
    evaluated trial's proposal margin and |1 - p_d/p_t - u|), final_kind [R]
    (0 greedy, 1 residual drawn explicitly, 2 bonus row, 3 residual that was
    empty, drawn from p_t instead, 4 residual kept by a trial) and trials [R]
    (residual trials evaluated).
    """
    tokens = to_i64(tokens)
    lens = to_i64(lens)
    target = to_f64(target)
    R, G1, V = target.shape
    G = G1 - 1
    req = np.arange(R) if requests is None else to_i64(requests)
    dl = None if tau == 0.0 else to_f64(draft_logits)
    accepted = np.zeros(R, dtype=np.int64)
    bonus = np.zeros(R, dtype=np.int64)
    acc_margin = np.full((R, G), np.nan)
    final_margin = np.zeros(R)
    final_kind = np.zeros(R, dtype=np.int64)
    trials = np.zeros(R, dtype=np.int64)
    for i in range(R):
        L = int(lens[i])
        rq = int(req[i])
        n = L
        if tau == 0.0:
            for j in range(1, L + 1):
                y = int(np.argmax(target[i, j - 1]))
                if tokens[i, j - 1] != y:
                    n = j - 1
                    break
            bonus[i] = int(np.argmax(target[i, n]))
            final_margin[i] = top2_margin(target[i, n])
            accepted[i] = n
            continue
        rejected = False
        for j in range(1, L + 1):
            lt = target[i, j - 1] / tau
            ld = dl[i, j - 1] / tau
            lse_t = logsumexp(lt)
            lse_d = logsumexp(ld)
            x = int(tokens[i, j - 1])
            u = float(philox.uniform(seed, j, rq, philox.STREAM_ACCEPT, 0))
            m = np.log(u) + (ld[x] - lse_d) - (lt[x] - lse_t)
            acc_margin[i, j - 1] = m
            if m < 0.0:                                  # u * p_d(x) < p_t(x)
                continue
            n = j - 1
            p_t = np.exp(lt - lse_t)
            p_d = np.exp(ld - lse_d)
            rejected = True
            # the residual by rejection from p_t: keep y_q iff u_q < 1 - p_d(y_q) / p_t(y_q)
            margin = np.inf
            for q in range(RESIDUAL_TRIALS):
                s = philox.STREAM_TRIAL0 + 8 * q
                prop = gumbel_max_trial(lt, seed, j, rq, s, block, TRIAL_SUPER)
                y = int(prop["token"])
                if y < 0:                                # no finite target entry
                    break
                trials[i] += 1
                uq = float(philox.uniform(seed, j, rq, s + 1, 0))
                keep = 1.0 - p_d[y] / p_t[y] - uq if p_t[y] > 0.0 else -np.inf
                margin = min(margin, prop["margin"], abs(keep))
                if keep > 0.0:
                    bonus[i] = y
                    final_kind[i] = 4
                    break
            if final_kind[i] == 4:
                final_margin[i] = margin
                break
            # no trial kept: the explicit residual, drawn by Gumbel-max
            qr = np.maximum(p_t - p_d, 0.0)
            with np.errstate(divide="ignore"):
                smp = gumbel_max(np.log(qr), seed, j, rq, philox.STREAM_RESIDUAL, block)
            final_kind[i] = 1
            if smp["token"][0] < 0:                      # empty residual: draw from p_t
                smp = gumbel_max(lt, seed, j, rq, philox.STREAM_RESIDUAL, block)
                final_kind[i] = 3
            bonus[i] = int(smp["token"][0])
            final_margin[i] = min(margin, smp["margin"][0])
            break
        if not rejected:
            smp = gumbel_max(target[i, L] / tau, seed, L + 1, rq, philox.STREAM_BONUS, block)
            bonus[i] = int(smp["token"][0])
            final_margin[i] = smp["margin"][0]
            final_kind[i] = 2
        accepted[i] = n
    return dict(accepted=accepted, bonus=bonus, accept_margin=acc_margin,
                final_margin=final_margin, final_kind=final_kind, trials=trials)


# ---------------------------------------------------------------------------
# one round, composed
# ---------------------------------------------------------------------------

def draft_round(inp: Dict, tau: float, seed: int, keep_logits: bool = False,
                forced=None) -> Dict[str, np.ndarray]:
    """a1-a4 on a workload's inputs (dict from workloads.make_inputs)."""
    base = base_logits(inp["h"], inp["W_lm"])
    out = markov_draft(base, inp["h"], inp["anchor"], inp["W1"], inp["W2"], inp["w_conf"],
                       inp["T"], tau, seed, forced=forced, keep_logits=keep_logits)
    out["base"] = base
    return out
