"""Plain, slow reference of the ForkAttention layer (test infrastructure only).

Sources (the five web pages collected for Flide; cited by page title and
section):
  * "Flide는 공유 상태를 정확히 분기해 결정 추론을 최대 9.5배 빠르게 한다"
    (onedev summary) - sections "어떻게 동작하나" (problem, eq. (1)),
    "무엇과 다른가" (stream, metadata, visibility, two-call GDN, Prop. 3.1),
    "어떻게 쓰나" (device metadata, checkpoint at m).
  * "Flide: Accelerating Decision Inference with Exact State Forking"
    (rainbus summary) - "前置知识" (readout formula, gated delta rule,
    short causal conv, TV distance), "核心方法", "方法步骤详情" (steps 1-4:
    stream order, visibility rule j_y=j_x, c_y in {0,c_x}, t_y<=t_x, window
    t_x-t_y<W, conv reads the trunk tail by index, checkpoint contents).

Readings where the pages are silent (each also listed in the design notes):
  R1 causal bound inclusive of self (t_y <= t_x);  R2 window keeps
  t_x - t_y < W;  R3 state S is d_v x d_k and o_t uses the updated S_t;
  R4 alpha, eta per token and per head;  R5 conv: depthwise over the q, k, v
  channels, no bias, tap K-1 multiplies the current token, zero history
  before position 0, SiLU after the conv;  R6 q and k are L2-normalised per
  head after conv+SiLU as x * (sum x^2 + 1e-6)^(-1/2);  R7 attention scale
  1/sqrt(d), rotary rotate-half pairs (i, i+d/2), angle t * theta^(-2i/d);
  R8 the readout input h_i is the GDN layer's output row of the question's
  last token, flattened over heads;  R9 the checkpoint at m holds the state
  after positions < m and the raw conv inputs of positions m-K+1..m-1.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence

import numpy as np

PAD = -1

# ----------------------------------------------------------------------------
# Metadata (onedev summary "무엇과 다른가"; rainbus "方法步骤详情" steps 1 and 3)
# ----------------------------------------------------------------------------


def split_desc(desc: np.ndarray, R: int, Nq: int):
    """Unpack [R trunk_len | R n_q | Nq q_len | R prefix_len | R ckpt_pos]."""
    d = np.asarray(desc, dtype=np.int64)
    P = d[0:R]
    n = d[R:2 * R]
    ql = d[2 * R:2 * R + Nq]
    pl = d[2 * R + Nq:3 * R + Nq]
    ck = d[3 * R + Nq:4 * R + Nq]
    return P, n, ql, pl, ck


def meta_ref(desc, R: int, Nq: int, T_cap: int, tile_tokens: int) -> Dict[str, np.ndarray]:
    """Per-token (j, c, t) metadata, segment table and work lists of a round.

    Stream order: every request's trunk tokens that are held in the stream
    (positions prefix_len..P-1), request after request, then every question,
    grouped by request in question order; pad rows only at the tail.  A
    question's positions continue from P.  Branch c = 0 is the trunk, c = i+1
    the i-th question of its request.

    Attention work list: per segment in table order, the segment is cut into
    tiles of ``tile_tokens`` tokens aligned to its start; tiles of one segment
    are listed from the last to the first.
    """
    P, n, ql, pl, ck = split_desc(desc, R, Nq)
    tok_req = [PAD] * T_cap
    tok_branch = [PAD] * T_cap
    tok_pos = [PAD] * T_cap
    seg = {k: [] for k in ("start", "len", "pos0", "req", "branch", "trunk_start", "trunk_len",
                           "state_idx")}
    req = {k: [] for k in ("trunk_len", "prefix_len", "prefix_off", "ckpt_pos", "trunk_start",
                           "first_q", "n_q")}
    x = 0
    trunk_start = []
    prefix_off = 0
    for j in range(R):
        trunk_start.append(x)
        Lj = int(P[j] - pl[j])
        for u in range(Lj):
            tok_req[x + u] = j
            tok_branch[x + u] = 0
            tok_pos[x + u] = int(pl[j]) + u
        seg["start"].append(x)
        seg["len"].append(Lj)
        seg["pos0"].append(int(pl[j]))
        seg["req"].append(j)
        seg["branch"].append(0)
        seg["trunk_start"].append(x)
        seg["trunk_len"].append(Lj)
        seg["state_idx"].append(j)
        req["trunk_len"].append(int(P[j]))
        req["prefix_len"].append(int(pl[j]))
        req["prefix_off"].append(prefix_off)
        req["ckpt_pos"].append(int(ck[j]))
        req["trunk_start"].append(x)
        req["n_q"].append(int(n[j]))
        prefix_off += int(pl[j])
        x += Lj
    q_last = []
    qi = 0
    for j in range(R):
        req["first_q"].append(qi)
        for c in range(int(n[j])):
            L = int(ql[qi])
            for u in range(L):
                tok_req[x + u] = j
                tok_branch[x + u] = c + 1
                tok_pos[x + u] = int(P[j]) + u
            seg["start"].append(x)
            seg["len"].append(L)
            seg["pos0"].append(int(P[j]))
            seg["req"].append(j)
            seg["branch"].append(c + 1)
            seg["trunk_start"].append(trunk_start[j])
            seg["trunk_len"].append(int(P[j] - pl[j]))
            seg["state_idx"].append(j)
            q_last.append(x + L - 1)
            x += L
            qi += 1
    T = x
    work_seg, work_off = [], []
    for s in range(len(seg["start"])):
        L = seg["len"][s]
        ntile = (L + tile_tokens - 1) // tile_tokens
        for t in range(ntile - 1, -1, -1):
            work_seg.append(s)
            work_off.append(t * tile_tokens)
    out = {"T": np.int64(T), "nseg": np.int64(len(seg["start"])),
           "tok_req": np.array(tok_req, dtype=np.int32),
           "tok_branch": np.array(tok_branch, dtype=np.int32),
           "tok_pos": np.array(tok_pos, dtype=np.int32),
           "q_last": np.array(q_last, dtype=np.int32),
           "work_seg": np.array(work_seg, dtype=np.int32),
           "work_off": np.array(work_off, dtype=np.int32)}
    for k, v in seg.items():
        out["seg_" + k] = np.array(v, dtype=np.int32)
    for k, v in req.items():
        out["req_" + k] = np.array(v, dtype=np.int32)
    return out


def visible(jx, cx, tx, jy, cy, ty, window: int = 0) -> bool:
    """Fork visibility of key y for query x (rainbus "方法步骤详情" step 2):
    same request, key in the trunk or the query's own branch, t_y <= t_x,
    and for a sliding-window layer t_x - t_y < W."""
    if jx != jy or jx < 0:
        return False
    if not (cy == 0 or cy == cx):
        return False
    if ty > tx:
        return False
    if window > 0 and tx - ty >= window:
        return False
    return True


# ----------------------------------------------------------------------------
# Rotary position embedding (onedev "무엇과 다른가": questions get the rotary
# positions they would have alone; reading R7 for the exact form)
# ----------------------------------------------------------------------------


def rope(x: np.ndarray, pos: np.ndarray, theta: float, dtype=np.float32) -> np.ndarray:
    """Rotate each head vector of x [L, H, d] by its token position.

    Pair (i, i + d/2) is rotated by the angle pos * theta^(-2i/d); the angle,
    cosine and sine are taken in float64, the rotation in ``dtype``.
    """
    L, H, d = x.shape
    half = d // 2
    inv = theta ** (-(2.0 * np.arange(half, dtype=np.float64)) / d)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :]
    c = np.cos(ang).astype(dtype)[:, None, :]
    s = np.sin(ang).astype(dtype)[:, None, :]
    x = x.astype(dtype)
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


# ----------------------------------------------------------------------------
# Attention over one isolated sequence (positions 0..L-1)
# ----------------------------------------------------------------------------


def attention_sequence(q, k, v, *, window: int = 0, rope_theta: float = 0.0, scale=None,
                       dtype=np.float32, rows: Optional[np.ndarray] = None,
                       row_block: int = 1024) -> np.ndarray:
    """Causal (optionally sliding-window) softmax attention of one sequence.

    q [L, Hq, d], k and v [L, Hkv, d]; q-head h reads kv-head h // (Hq/Hkv).
    For query row x the scores q_x . k_y * scale over keys y <= x (and
    x - y < W) are max-shifted, exponentiated and normalised; the output is
    the probability-weighted sum of v_y.  ``rows`` selects the query rows to
    return (all by default); rows are independent and computed in groups of
    ``row_block`` only to bound memory.
    """
    L, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    pos = np.arange(L)
    if rope_theta:
        qr = rope(q, pos, rope_theta, dtype)
        kr = rope(k, pos, rope_theta, dtype)
    else:
        qr = q.astype(dtype)
        kr = k.astype(dtype)
    vv = v.astype(dtype)
    rows = np.arange(L) if rows is None else np.asarray(rows)
    out = np.zeros((rows.shape[0], Hq, d), dtype=dtype)
    sc = dtype(scale)
    for b0 in range(0, rows.shape[0], row_block):
        rb = rows[b0:b0 + row_block]
        kmax = int(rb.max()) + 1
        y = np.arange(kmax)
        mask = y[None, :] <= rb[:, None]
        if window > 0:
            mask &= (rb[:, None] - y[None, :]) < window
        for h in range(Hq):
            g = h // G
            s = (qr[rb, h, :] @ kr[:kmax, g, :].T) * sc
            s = np.where(mask, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            p = np.exp(s - m)
            p = p / p.sum(axis=1, keepdims=True)
            out[b0:b0 + rb.shape[0], h, :] = p @ vv[:kmax, g, :]
    return out


# ----------------------------------------------------------------------------
# Gated DeltaNet over one isolated sequence (rainbus "前置知识": gated delta
# rule S_t = a_t S_{t-1}(I - e_t k_t k_t^T) + e_t v_t k_t^T, o_t = S_t q_t,
# preceded by a short causal convolution; readings R3-R6, R9)
# ----------------------------------------------------------------------------


def causal_conv(x: np.ndarray, w: np.ndarray, hist: Optional[np.ndarray] = None,
                dtype=np.float32) -> np.ndarray:
    """Depthwise causal conv: y_t[c] = sum_i w[c, i] * x_{t-K+1+i}[c].

    x [L, C] raw inputs; w [C, K]; ``hist`` [K-1, C] are the raw inputs of the
    K-1 positions before x (zeros: the sequence starts at position 0).
    """
    L, C = x.shape
    K = w.shape[1]
    if hist is None:
        hist = np.zeros((K - 1, C), dtype=dtype)
    xp = np.concatenate([hist.astype(dtype), x.astype(dtype)], axis=0)
    y = np.zeros((L, C), dtype=dtype)
    for i in range(K):
        y += w[:, i].astype(dtype)[None, :] * xp[i:i + L]
    return y


def silu(x: np.ndarray) -> np.ndarray:
    return x / (x.dtype.type(1) + np.exp(-x))


def l2norm(x: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """x * (sum x^2 + eps)^(-1/2) over the last axis."""
    return x / np.sqrt((x * x).sum(axis=-1, keepdims=True) + x.dtype.type(eps))


def gdn_inputs(q, k, v, conv_w, hist=None, dtype=np.float32):
    """Conv + SiLU over q, k, v, then L2-normalise q and k per head.

    q, k [L, H, dk], v [L, H, dv]; conv_w [3, H, d, K]; hist (optional)
    [K-1, 3, H, d] raw inputs before the sequence.  Returns (qh, kh, vh).
    """
    L, H, dk = q.shape
    dv = v.shape[2]
    outs = []
    for s, (x, dd) in enumerate(((q, dk), (k, dk), (v, dv))):
        xf = x.reshape(L, H * dd)
        wf = conv_w[s, :, :dd, :].reshape(H * dd, -1)
        hf = None if hist is None else hist[:, s, :, :dd].reshape(hist.shape[0], H * dd)
        y = silu(causal_conv(xf, wf, hf, dtype)).reshape(L, H, dd)
        outs.append(y)
    qh, kh, vh = outs
    return l2norm(qh), l2norm(kh), vh


def gdn_sequence(q, k, v, alpha, eta, conv_w, *, dtype=np.float32, S0=None, hist=None,
                 state_at: Sequence[int] = ()):
    """Token-by-token gated delta rule over one sequence.

    Per head: S <- a_t S - a_t e_t (S k_t) k_t^T + e_t v_t k_t^T, then
    o_t = S q_t (S is d_v x d_k; o uses the updated state).  ``S0``/``hist``
    start the sequence from a saved state and conv window (used only by the
    fork-structure pin; the literal runs start from zero).  Returns
    (o [L, H, dv], S_final [H, dv, dk], {t: state after t tokens}, window
    [K-1, 3, H, d] = raw inputs of the last K-1 positions).
    """
    L, H, dk = q.shape
    dv = v.shape[2]
    K = conv_w.shape[3]
    qh, kh, vh = gdn_inputs(q, k, v, conv_w, hist, dtype)
    a = alpha.astype(dtype)
    e = eta.astype(dtype)
    S = np.zeros((H, dv, dk), dtype=dtype) if S0 is None else S0.astype(dtype).copy()
    o = np.zeros((L, H, dv), dtype=dtype)
    states = {}
    want = set(int(t) for t in state_at)
    if 0 in want:
        states[0] = S.copy()
    for t in range(L):
        kt = kh[t]  # [H, dk]
        Sk = np.matmul(S, kt[:, :, None])[:, :, 0]  # [H, dv]
        at = a[t][:, None, None]
        et = e[t][:, None, None]
        S = at * S - (at * et) * (Sk[:, :, None] * kt[:, None, :]) + et * (vh[t][:, :, None] * kt[:, None, :])
        o[t] = np.matmul(S, qh[t][:, :, None])[:, :, 0]
        if (t + 1) in want:
            states[t + 1] = S.copy()
    dmax = max(dk, dv)
    raw = np.zeros((L + K - 1, 3, H, dmax), dtype=dtype)
    if hist is not None:
        raw[:K - 1] = hist
    raw[K - 1:, 0, :, :dk] = q
    raw[K - 1:, 1, :, :dk] = k
    raw[K - 1:, 2, :, :dv] = v
    window = raw[L:L + K - 1].copy()
    return o, S, states, window


def conv_window_at(q, k, v, m: int, K: int):
    """Raw conv inputs of positions m-K+1..m-1 (zeros before position 0)."""
    L, H, dk = q.shape
    dv = v.shape[2]
    dmax = max(dk, dv)
    w = np.zeros((K - 1, 3, H, dmax), dtype=np.float32)
    for i in range(K - 1):
        t = m - (K - 1) + i
        if 0 <= t < L:
            w[i, 0, :, :dk] = q[t]
            w[i, 1, :, :dk] = k[t]
            w[i, 2, :, :dv] = v[t]
    return w


# ----------------------------------------------------------------------------
# Selective readout, eq. (1) (onedev "어떻게 동작하나"; rainbus "前置知识")
# ----------------------------------------------------------------------------


def readout(h: np.ndarray, w: np.ndarray, off: np.ndarray, dtype=np.float32) -> np.ndarray:
    """p_i(o) = exp(w_o . h_i) / sum_{o' in O_i} exp(w_o' . h_i).

    h [Nq, D] (one row per question), w [sum O, D], off [Nq+1] CSR offsets.
    """
    h = h.astype(dtype)
    w = w.astype(dtype)
    p = np.zeros(w.shape[0], dtype=dtype)
    for i in range(h.shape[0]):
        a, b = int(off[i]), int(off[i + 1])
        z = w[a:b] @ h[i]
        z = np.exp(z - z.max())
        p[a:b] = z / z.sum()
    return p


# ----------------------------------------------------------------------------
# Selective readout with the final pointwise block on the question rows only
# (onedev "어떻게 쓰나": in the last layer the MLP and what follows run only on
# each question's last-token row, which changes no output).  The pages give no
# form for the block; reading R10: pre-norm SwiGLU MLP with a residual, then a
# final RMSNorm, then eq. (1); RMSNorm x * (mean x^2 + 1e-6)^(-1/2) * g; the
# two GEMM inputs (normalised row, gated activation) are stored as bfloat16
# as in a bf16 model; everything else in `dtype`.
# ----------------------------------------------------------------------------


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 values rounded to the nearest bfloat16 (ties to even), as float32."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    keep = (u >> 16) & 1
    r = ((u + 0x7FFF + keep) >> 16) << 16
    return (r & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def rms_norm(x: np.ndarray, g: np.ndarray, eps: float = 1e-6, dtype=np.float32) -> np.ndarray:
    x = x.astype(dtype)
    return x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + dtype(eps)) * g.astype(dtype)


def mlp_block(h: np.ndarray, g1, w_gate, w_up, w_down, dtype=np.float32) -> np.ndarray:
    """y = h + W_down (silu(W_gate n) * (W_up n)), n = bf16(rms_norm(h, g1)); rows independent."""
    n = round_to_bf16(rms_norm(h, g1, dtype=np.float32)).astype(dtype)
    gate = n @ w_gate.astype(dtype).T
    up = n @ w_up.astype(dtype).T
    a = round_to_bf16((silu(gate) * up).astype(np.float32)).astype(dtype)
    return h.astype(dtype) + a @ w_down.astype(dtype).T


def readout_mlp(h: np.ndarray, g1, w_gate, w_up, w_down, g2, w: np.ndarray, off: np.ndarray,
                dtype=np.float32) -> np.ndarray:
    """Eq. (1) on z = rms_norm(mlp_block(h), g2), h [Nq, D] the questions' last-token rows."""
    y = mlp_block(h, g1, w_gate, w_up, w_down, dtype)
    return readout(rms_norm(y, g2, dtype=dtype), w, off, dtype)


def total_variation(p: np.ndarray, r: np.ndarray, off: np.ndarray) -> np.ndarray:
    """TV(P, Q) = 1/2 sum |p - q| per question (rainbus "前置知识")."""
    return np.array([0.5 * np.abs(p[off[i]:off[i + 1]] - r[off[i]:off[i + 1]]).sum()
                     for i in range(off.shape[0] - 1)])


# ----------------------------------------------------------------------------
# Round level: every trunk and every s ⊕ q_i as its own sequence
# ----------------------------------------------------------------------------


class RoundView:
    """The stream-layout inputs of one round, as plain arrays.

    ``layers[name]`` holds float32 arrays in stream layout (rows [T_cap]);
    ``prefix[name]`` (optional) holds the trunk rows kept outside the stream
    (request j's rows at [prefix_off_j, prefix_off_j + prefix_len_j)).
    """

    def __init__(self, desc, R, Nq, T_cap, layers, prefix=None):
        self.desc = np.asarray(desc)
        self.R, self.Nq, self.T_cap = R, Nq, T_cap
        self.layers = layers
        self.prefix = prefix
        self.meta = meta_ref(desc, R, Nq, T_cap, 32)
        (self.P, self.n, self.ql, self.pl, self.ck) = split_desc(desc, R, Nq)

    def sequence_rows(self, name: str, field: str, j: int, qi: Optional[int]) -> np.ndarray:
        """Rows of the isolated sequence s_j (qi None) or s_j ⊕ q_qi."""
        m = self.meta
        parts = []
        plj = int(self.pl[j])
        if plj > 0:
            off = int(m["req_prefix_off"][j])
            parts.append(self.prefix[name][field][off:off + plj])
        ts = int(m["req_trunk_start"][j])
        parts.append(self.layers[name][field][ts:ts + int(self.P[j]) - plj])
        if qi is not None:
            s = self.R + qi
            st, L = int(m["seg_start"][s]), int(m["seg_len"][s])
            parts.append(self.layers[name][field][st:st + L])
        return np.concatenate(parts, axis=0)

    def questions_of(self, j: int) -> List[int]:
        f = int(self.meta["req_first_q"][j])
        return list(range(f, f + int(self.n[j])))


def run_attention(view: RoundView, name: str, *, window: int, rope_theta: float, dtype=np.float32,
                  questions: Optional[Sequence[int]] = None, trunks: Optional[Sequence[int]] = None,
                  trunk_rows: Optional[Dict[int, np.ndarray]] = None) -> np.ndarray:
    """Stream-layout output of one attention layer, from isolated sequences.

    Trunk rows come from running trunk j alone; question rows from running
    s_j ⊕ q_i alone and keeping its last |q_i| rows.  ``questions``/``trunks``
    restrict which segments are computed (others stay zero); ``trunk_rows``
    optionally restricts trunk query rows (positions) per request.
    """
    m = view.meta
    Hq, d = view.layers[name]["q"].shape[1:]
    out = np.zeros((view.T_cap, Hq, d), dtype=dtype)
    trunks = range(view.R) if trunks is None else trunks
    questions = range(view.Nq) if questions is None else questions
    for j in trunks:
        q = view.sequence_rows(name, "q", j, None)
        k = view.sequence_rows(name, "k", j, None)
        v = view.sequence_rows(name, "v", j, None)
        plj = int(view.pl[j])
        rows = np.arange(plj, q.shape[0])
        if trunk_rows is not None and j in trunk_rows:
            rows = np.asarray(trunk_rows[j])
        if rows.shape[0] == 0:
            continue
        o = attention_sequence(q, k, v, window=window, rope_theta=rope_theta, dtype=dtype, rows=rows)
        ts = int(m["req_trunk_start"][j])
        out[ts + rows - plj] = o
    for qi in questions:
        j = int(m["seg_req"][view.R + qi])
        q = view.sequence_rows(name, "q", j, qi)
        k = view.sequence_rows(name, "k", j, qi)
        v = view.sequence_rows(name, "v", j, qi)
        L = int(m["seg_len"][view.R + qi])
        rows = np.arange(q.shape[0] - L, q.shape[0])
        o = attention_sequence(q, k, v, window=window, rope_theta=rope_theta, dtype=dtype, rows=rows)
        st = int(m["seg_start"][view.R + qi])
        out[st:st + L] = o
    return out


def run_gdn(view: RoundView, name: str, *, dtype=np.float32,
            questions: Optional[Sequence[int]] = None, trunks: Optional[Sequence[int]] = None):
    """Stream-layout output of one GDN layer, from isolated sequences.

    Returns dict: o [T_cap, H, dv]; S_P [R, H, dv, dk] (state after the whole
    trunk); conv_win [R, K-1, 3, H, d] (raw inputs of the trunk's last K-1
    positions); S_ckpt / conv_ckpt for requests with a checkpoint position.
    Every sequence starts from the zero state at position 0, including
    resumed trunks (their prefix rows are run again).
    """
    m = view.meta
    lay = view.layers[name]
    H, dk = lay["q"].shape[1:]
    dv = lay["v"].shape[2]
    K = lay["conv_w"].shape[3]
    dmax = max(dk, dv)
    out = {"o": np.zeros((view.T_cap, H, dv), dtype=dtype),
           "S_P": np.zeros((view.R, H, dv, dk), dtype=dtype),
           "conv_win": np.zeros((view.R, K - 1, 3, H, dmax), dtype=dtype),
           "S_ckpt": np.zeros((view.R, H, dv, dk), dtype=dtype),
           "conv_ckpt": np.zeros((view.R, K - 1, 3, H, dmax), dtype=dtype)}
    trunks = range(view.R) if trunks is None else trunks
    questions = range(view.Nq) if questions is None else questions

    def seq(j, qi):
        return [view.sequence_rows(name, f, j, qi) for f in ("q", "k", "v", "alpha", "eta")]

    for j in trunks:
        q, k, v, a, e = seq(j, None)
        ck = int(view.ck[j])
        o, S, states, win = gdn_sequence(q, k, v, a, e, lay["conv_w"], dtype=dtype,
                                         state_at=[ck] if ck >= 0 else [])
        plj = int(view.pl[j])
        ts = int(m["req_trunk_start"][j])
        out["o"][ts:ts + q.shape[0] - plj] = o[plj:]
        out["S_P"][j] = S
        out["conv_win"][j] = win
        if ck >= 0:
            out["S_ckpt"][j] = states[ck]
            out["conv_ckpt"][j] = conv_window_at(q, k, v, ck, K)
    for qi in questions:
        j = int(m["seg_req"][view.R + qi])
        q, k, v, a, e = seq(j, qi)
        L = int(m["seg_len"][view.R + qi])
        o, _, _, _ = gdn_sequence(q, k, v, a, e, lay["conv_w"], dtype=dtype)
        st = int(m["seg_start"][view.R + qi])
        out["o"][st:st + L] = o[q.shape[0] - L:]
    return out


def run_readout(view: RoundView, h_stream: np.ndarray, w: np.ndarray, off: np.ndarray,
                dtype=np.float32) -> np.ndarray:
    """Eq. (1) at each question's last stream row of h (flattened heads)."""
    rows = view.meta["q_last"]
    h = h_stream[rows].reshape(rows.shape[0], int(np.prod(h_stream.shape[1:])))  # also for no question
    return readout(h, w, off, dtype)


# ----------------------------------------------------------------------------
# Token trees: branches that fork again (rainbus summary "未来方向" (2): a tree of
# draft tokens has the shape of a request tree and runs in the same flat
# stream).  Every node's result is that of its own sequence, its ancestors'
# tokens followed by its own, run from scratch: the exactness statement at
# every fork.
# ----------------------------------------------------------------------------


def run_tree(layers: Dict[str, Dict[str, np.ndarray]], parent: np.ndarray, node_len: np.ndarray,
             attn: Sequence[tuple], gdn_name: str, w: np.ndarray, off: np.ndarray, dtype=np.float32):
    """Outputs of a forest of token trees, node by node.

    layers[name][field]: float32 rows of all nodes, node after node; attn: (name,
    window, rope_theta) per attention layer.  Returns dict: "attn" {name: [T, Hq, d]},
    "gdn" [T, H, dv], "S_end" [N, H, dv, dk] (state after the node's last token),
    "p" (eq. (1) at each leaf's last token, leaves in node order).
    """
    N = parent.shape[0]
    start = np.concatenate([[0], np.cumsum(node_len)[:-1]]).astype(np.int64)
    T = int(node_len.sum())

    def chain(k):
        c = [k]
        while parent[c[-1]] >= 0:
            c.append(int(parent[c[-1]]))
        return c[::-1]

    def seq(name, field, k):
        return np.concatenate([layers[name][field][start[a]:start[a] + node_len[a]] for a in chain(k)], axis=0)

    out = {"attn": {}, "S_end": None}
    for name, window, theta in attn:
        Hq, d = layers[name]["q"].shape[1:]
        o_all = np.zeros((T, Hq, d), dtype=dtype)
        for k in range(N):
            L = int(node_len[k])
            if L == 0:
                continue
            q, kk, v = seq(name, "q", k), seq(name, "k", k), seq(name, "v", k)
            rows = np.arange(q.shape[0] - L, q.shape[0])
            o_all[start[k]:start[k] + L] = attention_sequence(q, kk, v, window=window, rope_theta=theta,
                                                              dtype=dtype, rows=rows)
        out["attn"][name] = o_all
    lay = layers[gdn_name]
    H, dk = lay["q"].shape[1:]
    dv = lay["v"].shape[2]
    o_all = np.zeros((T, H, dv), dtype=dtype)
    S_end = np.zeros((N, H, dv, dk), dtype=dtype)
    for k in range(N):
        q, kk, v, a, e = (seq(gdn_name, f, k) for f in ("q", "k", "v", "alpha", "eta"))
        o, S, _, _ = gdn_sequence(q, kk, v, a, e, lay["conv_w"], dtype=dtype)
        L = int(node_len[k])
        o_all[start[k]:start[k] + L] = o[q.shape[0] - L:]
        S_end[k] = S
    out["gdn"] = o_all
    out["S_end"] = S_end
    leaves = [k for k in range(N) if not np.any(parent == k)]
    last = np.array([start[k] + node_len[k] - 1 for k in leaves], dtype=np.int64)
    out["p"] = readout(o_all[last].reshape(len(leaves), -1), w, off, dtype)
    return out


# Pins of each oracle function (what ties it to something other than itself).
PINS = {
    "meta_ref": "hand-written arrays (tests/golden) + randomized property checks",
    "rope": "complex-multiplication form, norm preservation, relative-position invariance",
    "attention_sequence": "brute-force flat-stream mask (fork structure), single key, uniform scores",
    "causal_conv": "numpy.convolve per channel",
    "gdn_sequence": "literal matrix form, eta=0, delta-rule recall, orthonormal keys, resume==scratch",
    "readout": "scipy.special.softmax, |O|=1, equal logits, sum to one",
    "round_to_bf16": "bit patterns of hand-picked ties and carries; idempotent; exact for bf16 values",
    "rms_norm": "constant rows map to sign * g; unit mean square; scale invariance",
    "mlp_block": "W_down = 0 gives h; literal per-row loop in fp64; rows independent (selective = full)",
    "readout_mlp": "W_down = 0 and g2 = 1 reduce to eq. (1) on rms_norm(h)",
    "run_tree": "depth-1 trees equal the round oracle; a chain tree equals one sequence; node outputs "
                "do not depend on other branches",
}
