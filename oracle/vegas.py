"""Plain fp64 CPU oracle of verification-guided sparse self-speculative decoding.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline leg may use it.  It is deliberately slow and literal: every function
writes out the definition it follows, in float64, with numpy matrix products as
the only library step.  Nothing here blocks, fuses or reorders beyond that.

Source page: "Resumo Técnico: Vegas – Decodificação Auto-Especulativa com Atenção
Esparsa Guiada por Verificação" (gist.science summary of paper 2602.07223):

* Vegas §2, core mechanism, step 1 (verification phase): the target model runs a
  standard forward pass with *full* attention over the prefix and the draft chain,
  and computes the attention logits of every KV entry along the way.
* Vegas §2, step 2 (KV selection) and step 3 (draft phase): the critical entries found
  during verification form the sparse attention mask of the next draft phase.
* Vegas §2.A, selection formula: T = argmax over T ⊆ P, |T| = k of
  Σ_{t=1..γ+1} Σ_{h∈H} Σ_{i∈T} l^{(h)}_{ti}  (logits summed over draft rows and
  query heads, accepted and rejected tokens alike).
* Vegas §2.B, Collect-2-Query: aggregate only the first draft token and the bonus
  token, the two rows farthest apart in the chain.
* Vegas §3, kernel instrumentation: the logits are taken *before* the softmax.
* Vegas §3, sparse execution: the draft's attention is a paged kernel with a page
  size of one token, the selected token indices serving as page indices, i.e. an
  attention over an explicit list of gathered cache entries.
* Vegas §5, lossless quality: verification uses full attention, so it is exact
  attention, not an approximation.

Readings where the page is silent (each is listed with its reason in the design
notes): logits include the 1/sqrt(d) scale; one selection per sequence (and per
layer), shared by all KV heads; P is the prefix before the verify rows; ties go to
the lower position; k >= n selects everything; query head h reads KV head
floor(h / G); the draft attends T plus the draft tokens appended so far, the
current one included.

Array conventions (all float64 unless stated):
  q_verify  [R][H_q][d]     R = gamma + 1 verify rows (row gamma = bonus token)
  K, V      [n][H_kv][d]    prefix entries of one sequence
  k_new     [R][H_kv][d]    the verify rows' own keys / values
  q_draft   [H_q][d]        one draft step's query
"""
from __future__ import annotations

import numpy as np


# --------------------------------------------------------------------- helpers
def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly (bf16 is the top half of fp32)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _default_scale(d: int, scale: float | None) -> float:
    return 1.0 / np.sqrt(d) if not scale else float(scale)


def softmax_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float,
                      allowed: np.ndarray | None = None):
    """Scaled dot-product attention of query rows q [M][d] over K, V [n][d].

    logits l = (q K^T) * scale; p = exp(l - max l) / sum exp(...) over the allowed
    entries; o = p V.  Returns (o [M][d], p [M][n], l [M][n]).
    """
    logits = (q @ K.T) * scale
    if allowed is not None:
        logits = np.where(allowed, logits, -np.inf)
    mx = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - mx)
    p = e / e.sum(axis=1, keepdims=True)
    return p @ V, p, logits


def _heads(Hq: int, Hkv: int):
    if Hq % Hkv:
        raise ValueError("H_q must be a multiple of H_kv")
    G = Hq // Hkv
    return G, [h // G for h in range(Hq)]


# ------------------------------------------------------------- verification
def verify_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, k_new: np.ndarray,
                     v_new: np.ndarray, scale: float | None = None) -> np.ndarray:
    """Full attention of the R verify rows (Vegas §2 step 1; lossless, Vegas §5).

    Row t of head h attends every prefix entry 0..n-1 and the new rows u <= t
    (causal among the draft chain, itself included), on KV head floor(h/G).
    Returns O [R][H_q][d].
    """
    R, Hq, d = q.shape
    n, Hkv, _ = K.shape
    s = _default_scale(d, scale)
    _, g_of = _heads(Hq, Hkv)
    out = np.zeros((R, Hq, d))
    for h in range(Hq):
        g = g_of[h]
        keys = np.concatenate([K[:, g, :], k_new[:, g, :]], axis=0)      # [n + R][d]
        vals = np.concatenate([V[:, g, :], v_new[:, g, :]], axis=0)
        allowed = np.zeros((R, n + R), dtype=bool)
        allowed[:, :n] = True
        for t in range(R):
            allowed[t, n:n + t + 1] = True
        o, _, _ = softmax_attention(q[:, h, :], keys, vals, s, allowed)
        out[:, h, :] = o
    return out


def verify_logits(q: np.ndarray, K: np.ndarray, scale: float | None = None) -> np.ndarray:
    """Pre-softmax logits l^{(h)}_{t i} = q_{t,h} . k_{i, floor(h/G)} * scale of every
    prefix entry i (Vegas §2 step 1; "before the softmax", Vegas §3).  [R][H_q][n]."""
    R, Hq, d = q.shape
    n, Hkv, _ = K.shape
    s = _default_scale(d, scale)
    _, g_of = _heads(Hq, Hkv)
    L = np.empty((R, Hq, n))
    for h in range(Hq):
        L[:, h, :] = (q[:, h, :] @ K[:, g_of[h], :].T) * s
    return L


def aggregated_scores(q: np.ndarray, K: np.ndarray, rows, scale: float | None = None) -> np.ndarray:
    """Per-entry objective of the selection formula (Vegas §2.A):
    s_i = Σ_{t in rows} Σ_{h} l^{(h)}_{t i} for every prefix entry i.

    rows = all verify rows (the formula as printed) or the Collect-2-Query pair
    {0, gamma} (Vegas §2.B).  The verify rows' own keys are not in P."""
    L = verify_logits(q, K, scale)
    rows = sorted(set(int(t) for t in rows))
    if any(t < 0 or t >= q.shape[0] for t in rows):
        raise ValueError("row outside the verify chain")
    return L[rows].sum(axis=(0, 1))


def aggregated_scores_grouped(q: np.ndarray, K: np.ndarray, rows, scale: float | None = None) -> np.ndarray:
    """The per-entry objective of aggregated_scores, computed through the linearity of
    the dot product: summed over the rows and the query heads of KV head g, the logits
    of entry i equal scale * k_{i,g} . (the sum of those query vectors).  One n x d
    product per KV head instead of one per (row, query head); the full-size checks
    use it.  [n]."""
    R, Hq, d = q.shape
    n, Hkv, _ = K.shape
    s = _default_scale(d, scale)
    G, _ = _heads(Hq, Hkv)
    rows = sorted(set(int(t) for t in rows))
    if any(t < 0 or t >= R for t in rows):
        raise ValueError("row outside the verify chain")
    out = np.zeros(n)
    for g in range(Hkv):
        qsum = q[rows][:, g * G:(g + 1) * G, :].sum(axis=(0, 1))
        out += K[:, g, :] @ qsum
    return out * s


def select_topk(s: np.ndarray, k: int) -> np.ndarray:
    """The size-k subset maximising Σ_{i in T} s_i (Vegas §2.A's argmax).

    Because the objective is a sum of per-entry terms, a maximiser is any k entries
    with the largest s_i; among equal scores the lower position is preferred, which
    makes the set unique.  -0.0 is treated as +0.0.  k >= n selects every entry.
    Returns the chosen positions in ascending order (int64)."""
    s = np.asarray(s, dtype=np.float64) + 0.0          # -0.0 + 0.0 == +0.0
    n = s.shape[0]
    if k < 0:
        raise ValueError("k must be >= 0")
    m = min(k, n)
    order = np.lexsort((np.arange(n), -s))             # by score desc, then position asc
    return np.sort(order[:m]).astype(np.int64)


def select_window(n: int, k: int) -> np.ndarray:
    """The query-agnostic baseline of Vegas §1 (problem statement: sliding windows select
    cheaply but draft poorly): the last min(k, n) prefix positions, ascending (int64)."""
    if k < 0 or n < 0:
        raise ValueError("n and k must be >= 0")
    m = min(k, n)
    return np.arange(n - m, n, dtype=np.int64)


def selection_overlap(a: np.ndarray, b: np.ndarray, k: int) -> float:
    """|A ∩ B| / k: how much two selections agree (Vegas §2.B observation)."""
    if k <= 0:
        return 1.0
    return len(np.intersect1d(a, b)) / float(k)


# ------------------------------------------------------------------ paged cache
def paged_slots(table_row: np.ndarray, page_size: int, n: int) -> np.ndarray:
    """Physical slots of tokens 0..n-1 of one sequence in a paged cache (the block table
    of Vegas §3, whose draft kernel takes tokens as pages): token i lives in row
    i % page_size of page table_row[i // page_size], page p holding slots
    p * page_size .. p * page_size + page_size - 1.  int64 [n]."""
    i = np.arange(n, dtype=np.int64)
    return np.asarray(table_row, dtype=np.int64)[i // page_size] * page_size + i % page_size


# ------------------------------------------------------------------ drafting
def sparse_draft_attention(q: np.ndarray, K_sel: np.ndarray, V_sel: np.ndarray,
                           scale: float | None = None) -> np.ndarray:
    """Attention of one draft query q [H_q][d] over an explicit list of cache entries
    K_sel, V_sel [m][H_kv][d] (page size one, Vegas §3 sparse execution).  [H_q][d]."""
    Hq, d = q.shape
    m, Hkv, _ = K_sel.shape
    s = _default_scale(d, scale)
    _, g_of = _heads(Hq, Hkv)
    out = np.zeros((Hq, d))
    for h in range(Hq):
        o, _, _ = softmax_attention(q[h:h + 1, :], K_sel[:, g_of[h], :], V_sel[:, g_of[h], :], s)
        out[h] = o[0]
    return out


def draft_step(q: np.ndarray, K: np.ndarray, V: np.ndarray, idx: np.ndarray,
               tail_K: np.ndarray, tail_V: np.ndarray, scale: float | None = None) -> np.ndarray:
    """One sparse draft step (Vegas §2 step 3): attend the selected prefix entries
    idx (into K, V) plus the tail of draft tokens appended so far, tail_K/tail_V
    [s+1][H_kv][d], the current token last."""
    idx = np.asarray(idx, dtype=np.int64)
    K_sel = np.concatenate([K[idx], tail_K], axis=0)
    V_sel = np.concatenate([V[idx], tail_V], axis=0)
    return sparse_draft_attention(q, K_sel, V_sel, scale)


def iteration(q_verify, K, V, k_new, v_new, q_draft, k_draft, v_draft, k: int,
              rows0, rows1=None, scale: float | None = None, select_on=None) -> dict:
    """One verify -> select -> gamma-step draft round for one sequence.

    1. verify: full attention of the R rows (Vegas §2 step 1);
    2. scores on rows0 (and rows1) (Vegas §2.A / §2.B);
    3. T = top-k of the rows0 scores, or of ``select_on`` when the caller passes
       scores (the GPU's own, for a bit-exact index check);
    4. draft step s = 0..gamma-1: the draft token's K/V is appended after the prefix
       (slot n + s) and the query attends T plus draft tokens 0..s (Vegas §2 step 3).
    """
    gamma = q_draft.shape[0]
    O_v = verify_attention(q_verify, K, V, k_new, v_new, scale)
    s0 = aggregated_scores(q_verify, K, rows0, scale)
    s1 = aggregated_scores(q_verify, K, rows1, scale) if rows1 is not None else None
    T = select_topk(s0 if select_on is None else select_on, k)
    O_d = np.zeros((gamma,) + q_draft.shape[1:])
    for s in range(gamma):
        O_d[s] = draft_step(q_draft[s], K, V, T, k_draft[:s + 1], v_draft[:s + 1], scale)
    return dict(out_verify=O_v, scores0=s0, scores1=s1, idx=T, out_draft=O_d)


# ------------------------------------------------------------------ acceptance
# Vegas §2 step 1 (verification phase: the target's full-attention pass decides which
# draft tokens are accepted) and §5 (lossless quality: the output follows the target
# model's distribution).  The page names acceptance without spelling out the rule; the
# rule written here is the standard one of speculative decoding (greedy: a draft token
# survives if it is the target's most likely token; sampling: accept x with probability
# min(1, p(x) / q(x)), resample a rejection from the normalised excess max(0, p - q)).
# Layout: p_logits [gamma+1][V] (row t: the target's distribution for the token after t
# accepted drafts; row gamma: the bonus position), q_logits [gamma][V] (the draft's
# distribution of draft token t), draft tokens x [gamma].

def softmax(logits: np.ndarray) -> np.ndarray:
    """exp(l - max l) / sum exp(l - max l) along the last axis (float64)."""
    l = np.asarray(logits, dtype=np.float64)
    e = np.exp(l - l.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def sample_inverse_cdf(w: np.ndarray, u: float) -> int:
    """The smallest v with sum_{i <= v} w_i > u * sum_i w_i (weights >= 0, not all zero;
    a token of weight zero is never drawn).  u in [0, 1)."""
    c = np.cumsum(np.asarray(w, dtype=np.float64))
    return int(np.searchsorted(c, u * c[-1], side="right"))


def argmax_lowest(v: np.ndarray) -> int:
    """Position of the largest value; ties go to the lowest position."""
    v = np.asarray(v)
    return int(np.flatnonzero(v == v.max())[0])


def accept_greedy(p_logits: np.ndarray, x: np.ndarray) -> tuple[int, int]:
    """(accepted count a, next token): draft t is kept while x_t is the target's most
    likely token at row t; the next token is that most likely token at row a."""
    gamma = len(x)
    a = 0
    while a < gamma and int(x[a]) == argmax_lowest(p_logits[a]):
        a += 1
    return a, argmax_lowest(p_logits[a])


def accept_sample(p_logits: np.ndarray, q_logits: np.ndarray, x: np.ndarray, u: np.ndarray,
                  u_res: float) -> tuple[int, int]:
    """(accepted count a, next token) by speculative sampling.  Draft t is accepted iff
    u_t * q_t(x_t) < p_t(x_t).  At the first rejection a the next token is drawn from the
    excess max(0, p_a - q_a) (from p_a if that is zero everywhere); after gamma
    acceptances it is drawn from p_gamma; both by inverse CDF with u_res."""
    gamma = len(x)
    for t in range(gamma):
        p, q = softmax(p_logits[t]), softmax(q_logits[t])
        xt = int(x[t])
        if not (u[t] * q[xt] < p[xt]):
            w = np.maximum(0.0, p - q)
            return t, sample_inverse_cdf(w if w.sum() > 0 else p, u_res)
    return gamma, sample_inverse_cdf(softmax(p_logits[gamma]), u_res)


def next_prefix_len(n: int, a: int) -> int:
    """Prefix length after acceptance: the verified row before the drafts and the a
    accepted drafts enter the prefix (their keys and values are already in the cache)."""
    return n + a + 1
