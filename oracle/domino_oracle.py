"""Plain CPU oracle of the Domino draft-block rollout (fp64, numpy).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it.  It shares no code with the
CUDA library; it reads the seeded inputs (float32 arrays, or bf16 values as
raw uint16 bit patterns) and widens them itself.

What it computes (page "Add correctness-first Domino support to DFlash V2",
section "Design"; page "[Spec] Add Domino projector support to DFlash
speculative decoding (V2)", section "Implementation"):

  L[i, v]   = sum_h X[i, h] * W_lm[v, h]            base logits, all 16 rows
  p_1       = argmax_v L[rho(0), v]                 first proposal, uncorrected
  h         = GRU(emb[t_0], 0); h = GRU(emb[p_1], h)   two-token prefix
  for k = 1..14:
     z      = W1 h + s[k];  a = z * sigmoid(z)      projector layer 1 + SiLU
     c[v]   = W2[v] . a + b[v] + L[rho(k), v]       v in the candidate pool
     p_{k+1}= argmax_v c[v]
     if k < 14: h = GRU(emb[p_{k+1}], h)            feedback update
  rho(j)    = j + 1
  s[j]      = W_hid . X[rho(j)]  when s is not given (backbone half of layer 1)

Readings taken where the pages are silent (each is listed in the design notes
of the repository): rho(j) = j + 1 (block position 0 is the verified token);
h_0 = 0; GRU gate rows ordered r|z|n with PyTorch GRUCell algebra and no
biases; fc1 without bias; ties go to the lowest token id; the pool is the
top-K ids by max over the 15 used base rows (score descending, id ascending),
kept in ascending id order; K = 0 or K >= V means the full vocabulary.

Everything is computed in float64 from the exact input values.  All pins are
in ``tests/test_oracle_pins.py``; none is "unpinned" except the readings above,
which the pages do not fix (rho in particular).
"""
from __future__ import annotations

import numpy as np

BLOCK = 16
N_PROPOSALS = 15
N_CORRECTED = 14
ROW_OFFSET = 1  # rho(j) = j + ROW_OFFSET


def widen(x: np.ndarray) -> np.ndarray:
    """Exact float64 value of a float32 array or of raw bf16 bit patterns."""
    if x.dtype == np.uint16:
        f32 = (x.astype(np.uint32) << np.uint32(16)).view(np.float32)
        return f32.astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def silu(z):
    """SiLU(z) = z * sigmoid(z): the projector's activation (kernel text
    ``SiLU(z+s) @ fc2.T``, page "[Spec] Add Domino projector support",
    section "Implementation")."""
    return z * sigmoid(z)


def gru_cell(x, h, w_ih, w_hh):
    """One bias-free GRU update (PyTorch GRUCell algebra, gate rows r|z|n).

    Page "Add correctness-first Domino support to DFlash V2", section
    "Design": the prefix GRU is bias-free and ATen GRUCell does the one-token
    updates.  ``x`` [..., E], ``h`` [..., G]; ``w_ih`` [3G, E], ``w_hh`` [3G, G].
    """
    G = w_hh.shape[1]
    gi = x @ w_ih.T
    gh = h @ w_hh.T
    r = sigmoid(gi[..., 0:G] + gh[..., 0:G])
    u = sigmoid(gi[..., G:2 * G] + gh[..., G:2 * G])
    n = np.tanh(gi[..., 2 * G:3 * G] + r * gh[..., 2 * G:3 * G])
    return (1.0 - u) * n + u * h


def argmax_lowest(c: np.ndarray) -> int:
    """Index of the largest value; the lowest index among equal maxima."""
    return int(np.argmax(c))  # numpy returns the first maximal position


def top2_margin(c: np.ndarray) -> float:
    """c[top1] - c[top2] (0 when the maximum is tied, inf for one element)."""
    if c.shape[0] < 2:
        return float("inf")
    part = np.partition(c, -2)
    return float(part[-1] - part[-2])


def lm_head(X: np.ndarray, W_lm: np.ndarray, chunk: int = 16384) -> np.ndarray:
    """Base logits L[..., v] = sum_h X[..., h] W_lm[v, h] in float64.

    Page "support tensor-parallel Domino rollout", section "Rollout
    performance" (base LM-head over the block's draft hidden states) and page
    "Add correctness-first Domino support to DFlash V2", section "Design"
    (the base LM-head projection stays full-vocabulary).  ``W_lm`` may be raw
    bf16 bits; it is widened chunk by chunk to bound memory.
    """
    Xd = widen(X)
    V = W_lm.shape[0]
    out = np.empty(Xd.shape[:-1] + (V,), dtype=np.float64)
    for v0 in range(0, V, chunk):
        v1 = min(V, v0 + chunk)
        out[..., v0:v1] = Xd @ widen(W_lm[v0:v1]).T
    return out


def candidate_pool(L_rows: np.ndarray, K: int) -> np.ndarray:
    """Block-shared candidate pool of one request.

    Page "Add correctness-first Domino support to DFlash V2", section
    "Design": one per-request pool, shared by all steps of the block, K=0
    meaning the full vocabulary.  ``L_rows`` [15, V] are the base rows the
    proposals use; score[v] = max over them; the pool is the K ids with the
    largest score (ties to the lower id), returned in ascending id order.
    """
    V = L_rows.shape[1]
    if K <= 0 or K >= V:
        return np.arange(V, dtype=np.int64)
    score = L_rows.max(axis=0)
    order = np.lexsort((np.arange(V), -score))  # primary: score desc, then id asc
    return np.sort(order[:K])


def candidate_pool_compact(L_rows: np.ndarray, K: int, P: int) -> np.ndarray:
    """The same pool built the way the tensor-parallel stage C builds it.

    Page "feat: support tensor-parallel Domino rollout", section
    "Implementation", stage C: each of P ranks owns a contiguous vocabulary
    shard, takes its local top-K, and the P*K candidates are merged into the
    global top-K.  Shards are [p*S, min(V, (p+1)*S)) with S = ceil(V/P); both
    selections order by (score desc, id asc).  Returned in ascending id order.
    """
    V = L_rows.shape[1]
    if K <= 0 or K >= V:
        return np.arange(V, dtype=np.int64)
    score = L_rows.max(axis=0)
    S = -(-V // P)
    cand = []
    for p in range(P):
        lo, hi = p * S, min(V, (p + 1) * S)
        if lo >= hi:
            continue
        ids = np.arange(lo, hi)
        order = np.lexsort((ids, -score[lo:hi]))
        cand.append(ids[order[:K]])
    cand = np.concatenate(cand)
    order = np.lexsort((cand, -score[cand]))
    return np.sort(cand[order[:K]])


class OracleWeights:
    """Weights widened once to float64 (the analogue of load_weights)."""

    def __init__(self, w: dict):
        self.lm_head = w["lm_head"]  # kept in its input dtype, widened per chunk
        self.emb = widen(w["emb"])
        self.w_ih = widen(w["w_ih"])
        self.w_hh = widen(w["w_hh"])
        self.fc1 = widen(w["fc1"])
        self.fc2 = widen(w["fc2"])
        self.b = widen(w["b"])
        self.V = self.fc2.shape[0]
        self.G = self.w_hh.shape[1]
        self.F = self.fc1.shape[0]


def backbone_s(hidden, W_hid) -> np.ndarray:
    """Per-step additive term of projector layer 1 from the backbone hidden.

    The projector's first layer acts on the concatenation [backbone hidden |
    GRU state] (page "Add correctness-first Domino support to DFlash V2",
    the "add Domino drafter training backend" change: a low-rank embed_proj
    over [backbone hidden | GRU state]), so with W1 = [W_hid | fc1] it splits
    into W_hid . hidden + fc1 . h.  The term for proposal j uses the hidden
    state of the block row whose base logits that proposal corrects,
    rho(j) = j + 1.  Returns s [B, 15, F]:

        s[b, j, f] = sum_h hidden[b, rho(j), h] * W_hid[f, h]
    """
    X = widen(hidden)[:, ROW_OFFSET:ROW_OFFSET + N_PROPOSALS]   # [B,15,H]
    return np.einsum("bjh,fh->bjf", X, widen(W_hid))


def rollout(W: OracleWeights, hidden, s, verified, K: int = 0, forced=None,
            keep_scores: bool = False, n_proposals: int = N_PROPOSALS, W_hid=None) -> dict:
    """Run the Domino rollout for a batch of independent requests.

    ``hidden`` [B,16,H], ``s`` [B,15,F], ``verified`` [B] int.  ``forced``
    (optional [B,15] ints) teacher-forces the chain: the GRU is fed
    ``forced[:, k]`` instead of the rollout's own choice, while the rollout's
    own argmax is still reported in ``tokens``.

    ``s`` may be None when ``W_hid`` ([F, H], the backbone-hidden half of
    projector layer 1) is given: then s = backbone_s(hidden, W_hid).

    ``n_proposals`` (1..15) stops the chain after that many proposals, as
    for a target that verifies only the first n+1 block positions (page
    "feat: support tensor-parallel Domino rollout", section "Qwen3.6-27B
    checkpoint and full serving benchmark": b8 verifies 8 positions, n = 7,
    with the block-16 draft unchanged).  The draft is not shortened: the
    LM-head covers all 16 rows and the pool is still taken over rows 1..15.
    ``tokens`` entries from n on are -1; ``h``, ``z``, ``margin``, ``top1``
    keep their shapes with the unused entries left at zero.

    Returns a dict with ``tokens`` [B,15], ``L`` [B,16,V], ``pool`` (list of
    id arrays), ``h`` [B,15,G] (state after each of the 15 GRU updates),
    ``z`` [B,14,F] (pre-activation of each corrected step), ``margin`` [B,15]
    (top-1 minus top-2 score of every proposal), ``top1`` [B,15] (winning
    score) and, with ``keep_scores``, ``c`` (per request, [14, |pool|]).
    """
    if not 1 <= n_proposals <= N_PROPOSALS:
        raise ValueError("n_proposals must lie in 1..%d" % N_PROPOSALS)
    n_corr = n_proposals - 1
    B = hidden.shape[0]
    L = lm_head(hidden, W.lm_head)                     # [B,16,V]
    if s is None:
        if W_hid is None:
            raise ValueError("either s or W_hid is needed")
        s64 = backbone_s(hidden, W_hid)
    else:
        s64 = widen(s)
    tokens = np.zeros((B, N_PROPOSALS), dtype=np.int64)
    margin = np.zeros((B, N_PROPOSALS))
    top1 = np.zeros((B, N_PROPOSALS))
    hs = np.zeros((B, N_PROPOSALS, W.G))
    zs = np.zeros((B, N_CORRECTED, W.F))
    pools = []
    scores = []

    for r in range(B):
        rows = L[r, ROW_OFFSET:ROW_OFFSET + N_PROPOSALS]   # rho(0..14)
        pools.append(candidate_pool(rows, K))
        base0 = L[r, ROW_OFFSET]
        tokens[r, 0] = argmax_lowest(base0)
        margin[r, 0] = top2_margin(base0)
        top1[r, 0] = base0[tokens[r, 0]]
        scores.append([])

    def fed(r, j):
        return int(forced[r, j]) if forced is not None else int(tokens[r, j])

    # two-token prefix [verified, p_1], batched over requests
    h = np.zeros((B, W.G))
    h = gru_cell(W.emb[np.asarray(verified, dtype=np.int64)], h, W.w_ih, W.w_hh)
    hs[:, 0] = h
    h = gru_cell(W.emb[[fed(r, 0) for r in range(B)]], h, W.w_ih, W.w_hh)
    hs[:, 1] = h

    full = all(len(p) == W.V for p in pools)
    for k in range(1, n_corr + 1):
        z = h @ W.fc1.T + s64[:, k]
        zs[:, k - 1] = z
        a = silu(z)
        base = L[:, ROW_OFFSET + k]
        if full:
            c_all = a @ W.fc2.T + W.b + base                 # [B,V]
        for r in range(B):
            if full:
                c = c_all[r]
            else:
                p = pools[r]
                c = W.fc2[p] @ a[r] + W.b[p] + base[r, p]
            j = argmax_lowest(c)
            tokens[r, k] = pools[r][j]
            margin[r, k] = top2_margin(c)
            top1[r, k] = c[j]
            if keep_scores:
                scores[r].append(c.copy())
        if k < n_corr:
            h = gru_cell(W.emb[[fed(r, k) for r in range(B)]], h, W.w_ih, W.w_hh)
            hs[:, k + 1] = h

    tokens[:, n_proposals:] = -1
    out = {"tokens": tokens, "L": L, "pool": pools, "h": hs, "z": zs,
           "margin": margin, "top1": top1}
    if keep_scores:
        out["c"] = [np.stack(sc) if sc else np.zeros((0, len(p))) for sc, p in zip(scores, pools)]
    return out


def run(weights: dict, requests: dict, K: int = 0, **kw) -> dict:
    """Convenience wrapper: widen ``weights`` and run ``rollout``."""
    return rollout(OracleWeights(weights), requests["hidden"], requests.get("s"),
                   requests["verified"], K, **kw)
