"""fp64 CPU oracle of the block-diffusion MoE denoising step (test infrastructure only).

Sources, cited by page title and section:

* [AIT] the aitujian.cn engineering analysis of Clover-35B-A3B-Preview:
  section 二 (block diffusion: blocks are autoregressive between each other,
  parallel inside; block size 1 is ordinary autoregression), section 三 (the
  LowConfidence decode loop and its pseudo-code; the (1-p)^32 toy estimate),
  section 四 (40 layers, 256 routed experts, top-8, one shared expert per
  layer), section 五 (the union of experts touched by a 32-token block).
* [GRM] "What Is Clover-35B-A3B? Block Diffusion on a Qwen3.6 MoE" (goremy.ai):
  "How does confidence-threshold block decoding work?" and
  "What is the MoE coreset and why does it matter?".

Readings where the pages are silent or ambiguous (each is listed in the
design notes with its reason):

R1  The coreset aggregates each top-k candidate's full-softmax probability
    ("mass"), before any top-k renormalisation.
R2  Gates are the candidates' masses renormalised to sum to 1; after the
    coreset they are renormalised over the surviving candidates.  A token
    with no surviving candidate gets no routed output (the shared expert
    still applies).  Survivors whose masses are all zero also get zero gates.
R3  Expert ranking and top-k ties break toward the lower expert index; the
    top-k is ranked on the router logit, not on the rounded probability.
R4  Coreset arithmetic is exact: each fp32 mass is turned into the integer
    rne(mass * 2^54), sums are integer, the target is
    ceil(fp32(top_p) * double(total)) clamped to [1, total]; the selection is
    the shortest prefix of the ranking whose cumulative sum reaches the
    target.  top_p >= 1 (or an all-zero total) selects every candidate.
R5  The commit threshold test is conf >= threshold.
R6  Acceptance and the fallback range over still-masked positions only; a
    committed token is never rewritten.  Fallback ties go to the lowest
    position; argmax ties to the lowest token id.
R7  The shared expert is added with weight 1.
R8  Between MoE layers the stack is pre-norm residual with RMSNorm
    (gamma = 1, eps = 1e-6); the LM head reads RMSNorm of the final residual.
R9  In bf16 configurations the tensor a layer consumes (its normalised input
    and the LM-head input) is a bf16 tensor: the oracle rounds it to bf16
    (nearest-even) exactly where the model hands it over, then computes in
    float64.  Nothing else is rounded.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Callable, Sequence

import numpy as np

__all__ = [
    "round_bf16", "router_logits", "softmax", "topk_by_logit", "route", "route_from_logits",
    "mass_to_fixed", "coreset_select", "silu", "swiglu_expert", "moe_ffn", "plain_topk_moe",
    "rmsnorm", "lm_logits", "confidence_and_choice", "lowconfidence_commit", "block_decode_step",
    "MoELayer", "tiny_model_logits", "lowconfidence_loop", "CoresetResult", "CommitResult",
]


# ----------------------------------------------------------------------------------------------
# precision helper (R9)
# ----------------------------------------------------------------------------------------------
def round_bf16(v: np.ndarray) -> np.ndarray:
    """Round to the nearest bfloat16 (ties to even) and return float64.

    Goes through binary32 first; for values already representable in binary32
    that first step is exact, and the bf16 step rounds the 16 low mantissa bits.
    """
    f = np.asarray(v, dtype=np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16 << 16
    return (b.astype(np.uint32)).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------------------------
# (a1) router: logits, softmax, top-k        [AIT 四], [GRM "What is the MoE coreset ..."]
# ----------------------------------------------------------------------------------------------
def router_logits(x: np.ndarray, Wr: np.ndarray) -> np.ndarray:
    """z[t, e] = sum_h x[t, h] * Wr[e, h], in float64."""
    return np.asarray(x, np.float64) @ np.asarray(Wr, np.float64).T


def softmax(z: np.ndarray) -> np.ndarray:
    """Row softmax with the row maximum subtracted first."""
    z = np.asarray(z, np.float64)
    e = np.exp(z - z.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def topk_by_logit(z: np.ndarray, k: int) -> np.ndarray:
    """Per row, the k expert ids with the largest logits; ties to the lower id (R3)."""
    z = np.asarray(z, np.float64)
    T, E = z.shape
    ids = np.arange(E)
    out = np.empty((T, k), np.int32)
    for t in range(T):
        order = np.lexsort((ids, -z[t]))  # primary key -z (descending z), then id ascending
        out[t] = order[:k]
    return out


def route_from_logits(z: np.ndarray, k: int):
    """Top-k, masses and gates from given router logits.

    mass[t, j] = softmax(z[t])[idx[t, j]] (R1); gate = mass / sum_j mass (R2).
    """
    idx = topk_by_logit(z, k)
    p = softmax(z)
    mass = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    gate = mass / mass.sum(axis=1, keepdims=True)
    return idx, mass, gate


def route(x: np.ndarray, Wr: np.ndarray, k: int):
    """Router of one MoE layer: returns (idx, mass, gate, logits)."""
    z = router_logits(x, Wr)
    idx, mass, gate = route_from_logits(z, k)
    return idx, mass, gate, z


# ----------------------------------------------------------------------------------------------
# (a2) block coreset                          [GRM "What is the MoE coreset and why does it matter?"]
# ----------------------------------------------------------------------------------------------
FIXED_SHIFT = 54


def mass_to_fixed(mass) -> np.ndarray:
    """R4: integer rne(fp32(mass) * 2^54).  The product is exact in float64."""
    m32 = np.asarray(mass, np.float32).astype(np.float64)
    return np.rint(m32 * float(2 ** FIXED_SHIFT)).astype(np.int64)


@dataclass
class CoresetResult:
    n_sel: np.ndarray      # [R] int32, number of experts kept per request
    sel: list              # R lists of expert ids in ranking order (length n_sel[r])
    survive: np.ndarray    # [T, k] bool
    gate_rr: np.ndarray    # [T, k] float64, 0 where not surviving
    ranking: list          # R lists: every candidate expert in ranking order
    agg: list              # R dicts expert -> integer aggregated mass
    target: list           # R integer targets (None when everything is kept)


def coreset_select(idx: np.ndarray, mass: np.ndarray, top_p: Sequence[float] | float,
                   tokens_per_req: int) -> CoresetResult:
    """Block coreset per request (a block of `tokens_per_req` consecutive tokens).

    For each request: sum every top-k candidate's mass per expert over the
    block, rank experts by that sum (descending; ties to the lower id), keep
    the shortest prefix of the ranking that covers top_p of the summed mass,
    then restrict each token to its candidates inside the kept set and
    renormalise its gates over them (R1, R2, R4).
    """
    idx = np.asarray(idx)
    mass = np.asarray(mass, np.float64)
    T, k = idx.shape
    if T % tokens_per_req:
        raise ValueError("T must be a multiple of tokens_per_req")
    R = T // tokens_per_req
    tps = [top_p] * R if np.isscalar(top_p) else list(top_p)
    q = mass_to_fixed(mass)
    survive = np.zeros((T, k), bool)
    gate_rr = np.zeros((T, k), np.float64)
    n_sel = np.zeros(R, np.int32)
    sels, rankings, aggs, targets = [], [], [], []
    for r in range(R):
        rows = range(r * tokens_per_req, (r + 1) * tokens_per_req)
        agg: dict[int, int] = {}
        for t in rows:
            for j in range(k):
                e = int(idx[t, j])
                agg[e] = agg.get(e, 0) + int(q[t, j])   # Python ints: exact
        ranking = sorted(agg, key=lambda e: (-agg[e], e))
        total = sum(agg.values())
        tp = float(np.float32(tps[r]))
        if not (tp > 0.0):
            raise ValueError("top_p must be > 0")
        if tp >= 1.0 or total == 0:
            m, target = len(ranking), None
        else:
            target = math.ceil(tp * float(total))
            target = min(max(target, 1), total)
            cum, m = 0, 0
            for e in ranking:
                cum += agg[e]
                m += 1
                if cum >= target:
                    break
        keep = set(ranking[:m])
        for t in rows:
            s = [int(idx[t, j]) in keep for j in range(k)]
            survive[t] = s
            denom = sum(mass[t, j] for j in range(k) if s[j])
            for j in range(k):
                gate_rr[t, j] = mass[t, j] / denom if (s[j] and denom > 0.0) else 0.0
        n_sel[r] = m
        sels.append(ranking[:m])
        rankings.append(ranking)
        aggs.append(agg)
        targets.append(target)
    return CoresetResult(n_sel, sels, survive, gate_rr, rankings, aggs, targets)


# ----------------------------------------------------------------------------------------------
# (a3-a5) routed + shared SwiGLU experts      [AIT 四, 五], [GRM "How does Clover turn ..."]
# ----------------------------------------------------------------------------------------------
def silu(a: np.ndarray) -> np.ndarray:
    """silu(a) = a / (1 + exp(-a))."""
    a = np.asarray(a, np.float64)
    with np.errstate(over="ignore"):
        return a / (1.0 + np.exp(-a))


def swiglu_expert(x: np.ndarray, Wg: np.ndarray, Wu: np.ndarray, Wd: np.ndarray) -> np.ndarray:
    """y = Wd (silu(Wg x) * (Wu x)) for each row x; Wg, Wu: [I, H], Wd: [H, I]."""
    x = np.asarray(x, np.float64)
    g = x @ np.asarray(Wg, np.float64).T
    u = x @ np.asarray(Wu, np.float64).T
    return (silu(g) * u) @ np.asarray(Wd, np.float64).T


@dataclass
class MoELayer:
    """Weights of one MoE layer as float64 accessors.

    Wr: [E, H]; expert(e) -> (Wg [I, H], Wu [I, H], Wd [H, I]);
    shared() -> (Wg [Is, H], Wu [Is, H], Wd [H, Is]).
    """
    Wr: np.ndarray
    expert: Callable[[int], tuple]
    shared: Callable[[], tuple]


def moe_ffn(x: np.ndarray, layer: MoELayer, idx: np.ndarray, gate_rr: np.ndarray) -> np.ndarray:
    """out[t] = sum_j gate_rr[t, j] * y_{idx[t, j]}(x_t) + y_shared(x_t)   (R2, R7).

    Computed per expert over the tokens that use it, i.e. each expert's weights
    are applied to every block token routed to it.
    """
    x = np.asarray(x, np.float64)
    T, k = idx.shape
    out = np.zeros_like(x)
    users: dict[int, list] = {}
    for t in range(T):
        for j in range(k):
            if gate_rr[t, j] != 0.0:
                users.setdefault(int(idx[t, j]), []).append((t, j))
    for e in sorted(users):
        Wg, Wu, Wd = layer.expert(e)
        toks = [t for t, _ in users[e]]
        y = swiglu_expert(x[toks], Wg, Wu, Wd)
        for row, (t, j) in enumerate(users[e]):
            out[t] += gate_rr[t, j] * y[row]
    out += swiglu_expert(x, *layer.shared())
    return out


def plain_topk_moe(x: np.ndarray, layer: MoELayer, k: int) -> np.ndarray:
    """Ordinary per-token top-k MoE with a shared expert (what a block of one token must equal).

    Written independently of route/coreset: per token, rank logits, take the
    top k, weight the experts by a softmax over just those k logits.
    """
    x = np.asarray(x, np.float64)
    out = np.zeros_like(x)
    Wr = np.asarray(layer.Wr, np.float64)
    for t in range(x.shape[0]):
        z = Wr @ x[t]
        top = sorted(range(len(z)), key=lambda e: (-z[e], e))[:k]
        w = np.exp(np.array([z[e] for e in top]) - max(z[e] for e in top))
        w /= w.sum()
        for wj, e in zip(w, top):
            out[t] += wj * swiglu_expert(x[t:t + 1], *layer.expert(e))[0]
        out[t] += swiglu_expert(x[t:t + 1], *layer.shared())[0]
    return out


def rmsnorm(h: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """h / sqrt(mean(h^2) + eps) per row, gamma = 1 (R8)."""
    h = np.asarray(h, np.float64)
    return h / np.sqrt((h * h).mean(axis=-1, keepdims=True) + eps)


# ----------------------------------------------------------------------------------------------
# (a7-a8) LM head, confidence, LowConfidence commit        [AIT 三], [GRM "How does ... decoding work?"]
# ----------------------------------------------------------------------------------------------
def lm_logits(hidden: np.ndarray, Wlm: np.ndarray, scale: float = 1.0) -> np.ndarray:
    """logits[p, v] = scale * sum_h hidden[p, h] * Wlm[v, h]."""
    return scale * (np.asarray(hidden, np.float64) @ np.asarray(Wlm, np.float64).T)


def confidence_and_choice(logits: np.ndarray):
    """conf = max_v softmax(logits)[v] = 1 / sum_v exp(l_v - max l); choice = lowest argmax (R6)."""
    L = np.asarray(logits, np.float64)
    m = L.max(axis=1, keepdims=True)
    conf = 1.0 / np.exp(L - m).sum(axis=1)
    choice = np.argmax(L, axis=1).astype(np.int32)   # numpy returns the first maximum
    return conf, choice


@dataclass
class CommitResult:
    tokens: np.ndarray       # [R*P] int32 after the round
    masked: np.ndarray       # [R*P] bool after the round
    accept: np.ndarray       # [R*P] bool: committed in this round (threshold or fallback)
    fallback: np.ndarray     # [R] bool: the round used the single-position fallback
    n_committed: np.ndarray  # [R] int32


def lowconfidence_commit(conf, choice, tokens, masked, threshold: float, P: int) -> CommitResult:
    """One LowConfidence round for R requests of P positions each (R5, R6).

    Every still-masked position with conf >= threshold takes its choice; if
    none qualifies, the single most confident masked position does; positions
    already committed are left untouched.
    """
    conf = np.asarray(conf, np.float64)
    tokens = np.array(tokens, np.int32, copy=True)
    masked = np.array(masked, bool, copy=True)
    N = tokens.shape[0]
    R = N // P
    accept = np.zeros(N, bool)
    fallback = np.zeros(R, bool)
    n_comm = np.zeros(R, np.int32)
    for r in range(R):
        pos = [r * P + p for p in range(P) if masked[r * P + p]]
        if not pos:
            continue
        hit = [p for p in pos if conf[p] >= threshold]
        if not hit:
            best = pos[0]
            for p in pos[1:]:
                if conf[p] > conf[best]:
                    best = p
            hit = [best]
            fallback[r] = True
        for p in hit:
            tokens[p] = choice[p]
            masked[p] = False
            accept[p] = True
        n_comm[r] = len(hit)
    return CommitResult(tokens, masked, accept, fallback, n_comm)


# ----------------------------------------------------------------------------------------------
# whole step over the MoE stack, and the tiny embed -> MoE -> LM-head model
# ----------------------------------------------------------------------------------------------
def block_decode_step(h0, layers: Sequence[MoELayer], Wlm, top_p, k: int, tokens_per_req: int,
                      threshold: float, tokens, masked, bf16: bool, logit_scale: float = 1.0,
                      trace: list | None = None):
    """One denoising round of the MoE stack (mixers omitted) plus the commit.

    h_{l+1} = h_l + MoE_l(x_l), x_l = RMSNorm(h_l) (bf16-rounded when bf16, R9);
    hidden = RMSNorm(h_L) (bf16-rounded when bf16); then LM head, confidence
    and the LowConfidence commit.  Returns (h_L, hidden, logits, conf, choice,
    CommitResult).  `trace`, if given, receives per-layer dicts (x, idx, mass,
    coreset, out) for diagnosis.
    """
    q = round_bf16 if bf16 else (lambda v: np.asarray(v, np.float64))
    h = np.array(h0, np.float64, copy=True)
    for layer in layers:
        x = q(rmsnorm(h))
        idx, mass, _, z = route(x, layer.Wr, k)
        cs = coreset_select(idx, mass, top_p, tokens_per_req)
        out = moe_ffn(x, layer, idx, cs.gate_rr)
        if trace is not None:
            trace.append(dict(x=x, z=z, idx=idx, mass=mass, coreset=cs, out=out))
        h = h + out
    hidden = q(rmsnorm(h))
    logits = lm_logits(hidden, Wlm, logit_scale)
    conf, choice = confidence_and_choice(logits)
    res = lowconfidence_commit(conf, choice, tokens, masked, threshold, tokens_per_req)
    return h, hidden, logits, conf, choice, res


def tiny_model_logits(tokens, masked, emb, pos, layer: MoELayer, Wlm, top_p, k: int,
                      mask_id: int, logit_scale: float):
    """The one-layer embed -> MoE -> LM-head model that drives the full round loop.

    Input of position p: emb[mask_id] if p is masked, else emb[tokens[p]], plus
    pos[p % P].  Then the same pre-norm MoE layer and LM head as the stack.
    """
    tokens = np.asarray(tokens)
    P = pos.shape[0]
    ids = np.where(np.asarray(masked, bool), mask_id, tokens)
    h0 = np.asarray(emb, np.float64)[ids] + np.asarray(pos, np.float64)[np.arange(len(ids)) % P]
    x = rmsnorm(h0)
    idx, mass, _, _ = route(x, layer.Wr, k)
    cs = coreset_select(idx, mass, top_p, P)
    h = h0 + moe_ffn(x, layer, idx, cs.gate_rr)
    return lm_logits(rmsnorm(h), Wlm, logit_scale)


def lowconfidence_loop(logits_fn: Callable, n_pos: int, P: int, threshold: float,
                       max_steps: int | None = None):
    """Decode one block per request to resolution ([AIT 三], [GRM decoding loop]).

    logits_fn(tokens, masked, round) -> logits [n_pos, V].  All positions start
    masked; each round commits per `lowconfidence_commit`; stops when nothing is
    masked or after max_steps (default P) rounds.  Returns (tokens, rounds, history)
    where history holds each round's CommitResult.
    """
    tokens = np.zeros(n_pos, np.int32)
    masked = np.ones(n_pos, bool)
    steps = P if max_steps is None else max_steps
    history = []
    for rnd in range(steps):
        logits = logits_fn(tokens, masked, rnd)
        conf, choice = confidence_and_choice(logits)
        res = lowconfidence_commit(conf, choice, tokens, masked, threshold, P)
        history.append(res)
        tokens, masked = res.tokens, res.masked
        if not masked.any():
            break
    return tokens, len(history), history
