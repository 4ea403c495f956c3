"""ctypes wrapper of the plain CPU oracle (oracle/sdv_oracle.c, oracle/exact.c).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  It shares no
code with the CUDA library; both take their inputs from
``draft_verification_row_gb300.workloads``.

Every function takes numpy arrays (or CPU torch tensors) laid out exactly as
the CUDA library's arguments and returns numpy arrays.
"""
import ctypes
import numpy as np

from . import build as _build

MODE = {"token": 0, "greedy": 1, "block": 2, "multidraft": 3, "kseq": 4}
F32, BF16, F64 = 0, 1, 2
REQ_BAD_LENGTH, REQ_BAD_TOKEN, REQ_NONFINITE = 1, 2, 4
MAX_K = 16
MAX_L = 16


class _Problem(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("K", ctypes.c_int), ("L", ctypes.c_int), ("V", ctypes.c_int),
        ("row_stride", ctypes.c_longlong), ("dtype", ctypes.c_int),
        ("temperature", ctypes.c_double),
        ("target", ctypes.c_void_p), ("draft", ctypes.c_void_p),
        ("tokens", ctypes.c_void_p), ("lengths", ctypes.c_void_p),
        ("accept_u", ctypes.c_void_p), ("sample_u", ctypes.c_void_p),
    ]


class _TraceEntry(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("index", ctypes.c_int),
                ("lo", ctypes.c_double), ("hi", ctypes.c_double)]


class _Trace(ctypes.Structure):
    _fields_ = [("e", ctypes.POINTER(_TraceEntry)), ("cap", ctypes.c_int), ("n", ctypes.c_int)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(_build.build())
        _lib.sdvo_verify.restype = ctypes.c_int
        _lib.sdvo_exact_outcomes.restype = ctypes.c_int
        _lib.sdvo_exact_streams.restype = ctypes.c_int
        _lib.sdvo_exact_accept_len.restype = ctypes.c_int
        _lib.sdvo_prefix_index.restype = ctypes.c_longlong
        _lib.sdvo_sample_rows.restype = ctypes.c_int
        _lib.sdvo_lm_head_logits.restype = ctypes.c_int
    return _lib


def _np(a):
    """numpy view of a numpy array or CPU torch tensor (bf16 -> uint16 bits)."""
    if a is None:
        return None
    if hasattr(a, "detach"):
        import torch
        t = a.detach()
        if t.device.type != "cpu":
            raise ValueError("oracle inputs must be host tensors")
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        a = t.contiguous().numpy()
    return np.ascontiguousarray(a)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Problem:
    """One batch in the CUDA library's layout, held as numpy arrays."""

    def __init__(self, target, draft, tokens, lengths, accept_u, sample_u, temperature,
                 V=None):
        self.target = _np(target)
        self.draft = _np(draft)
        self.tokens = np.ascontiguousarray(_np(tokens), dtype=np.int32)
        self.lengths = None if lengths is None else np.ascontiguousarray(_np(lengths), dtype=np.int32)
        # uniforms are passed to the oracle as doubles (exact widening of fp32)
        self.accept_u = None if accept_u is None else np.ascontiguousarray(_np(accept_u), dtype=np.float64)
        self.sample_u = None if sample_u is None else np.ascontiguousarray(_np(sample_u), dtype=np.float64)
        self.temperature = float(temperature)
        t = self.target
        self.B, self.K = t.shape[0], t.shape[1]
        self.L = t.shape[2] - 1
        self.row_stride = t.shape[3]
        self.V = self.row_stride if V is None else int(V)
        if t.dtype in (np.uint16, np.int16):
            self.dtype = BF16
        elif t.dtype == np.float32:
            self.dtype = F32
        elif t.dtype == np.float64:
            self.dtype = F64
        else:
            raise TypeError(f"unsupported logit dtype {t.dtype}")

    def struct(self):
        s = _Problem()
        s.B, s.K, s.L, s.V = self.B, self.K, self.L, self.V
        s.row_stride = self.row_stride
        s.dtype = self.dtype
        s.temperature = self.temperature
        s.target, s.draft = _ptr(self.target), _ptr(self.draft)
        s.tokens, s.lengths = _ptr(self.tokens), _ptr(self.lengths)
        s.accept_u, s.sample_u = _ptr(self.accept_u), _ptr(self.sample_u)
        return s

    def request(self, b):
        """The same problem restricted to request b (a contiguous slab)."""
        return self.requests(b, b + 1)

    def requests(self, lo, hi):
        """The same problem restricted to requests lo..hi-1 (views, no copy)."""
        sub = object.__new__(Problem)
        sub.__dict__.update(self.__dict__)
        sl = slice(lo, hi)
        sub.target = self.target[sl]
        sub.draft = None if self.draft is None else self.draft[sl]
        sub.tokens = self.tokens[sl]
        sub.lengths = None if self.lengths is None else self.lengths[sl]
        sub.accept_u = None if self.accept_u is None else self.accept_u[sl]
        sub.sample_u = None if self.sample_u is None else self.sample_u[sl]
        sub.B = hi - lo
        return sub


def verify(mode, prob: Problem, residual_out=False, trace_cap=0):
    """Run the oracle; returns a dict of numpy arrays (and 'trace' if asked)."""
    B, K, L, V = prob.B, prob.K, prob.L, prob.V
    out = {
        "accept_len": np.zeros(B, np.int32),
        "accept_draft": np.zeros(B, np.int32),
        "out_token": np.zeros(B, np.int32),
        "accept_prob": np.zeros((B, K, L), np.float32),
        "residual_mass": np.zeros(B, np.float64),
        "margin": np.zeros(B, np.float64),
        "req_status": np.zeros(B, np.int32),
    }
    ro = np.zeros((B, V), np.float64) if residual_out else None
    tr = None
    entries = None
    if trace_cap:
        entries = (_TraceEntry * trace_cap)()
        tr = _Trace(ctypes.cast(entries, ctypes.POINTER(_TraceEntry)), trace_cap, 0)
    s = prob.struct()
    rc = lib().sdvo_verify(
        ctypes.c_int(MODE[mode]), ctypes.byref(s),
        _ptr(out["accept_len"]), _ptr(out["accept_draft"]), _ptr(out["out_token"]),
        _ptr(out["accept_prob"]), _ptr(out["residual_mass"]), _ptr(out["margin"]),
        _ptr(ro), _ptr(out["req_status"]), ctypes.byref(tr) if tr is not None else None)
    out["rc"] = rc
    if ro is not None:
        out["residual_out"] = ro
    if tr is not None:
        out["trace"] = [(entries[i].kind, entries[i].index, entries[i].lo, entries[i].hi)
                        for i in range(min(tr.n, trace_cap))]
    return out


def trace_counts(prob: Problem, trace, margin=1e-5):
    """Per request: the decisions the oracle took (comparisons of a uniform
    with a threshold, and inverse-CDF draws) and how many of them were
    within `margin` of flipping: |u - threshold| for an accept test, the
    distance of u to the ends of the chosen token's CDF interval for a draw.
    Returns two int arrays of shape [B]."""
    K, L = prob.K, prob.L
    dec = np.zeros(prob.B, np.int64)
    near = np.zeros(prob.B, np.int64)
    au = None if prob.accept_u is None else prob.accept_u.reshape(-1)
    su = None if prob.sample_u is None else prob.sample_u.reshape(-1)
    for kind, idx, lo, hi in trace:
        if kind == 0:
            b, m = idx // (K * L), abs(au[idx] - lo)
        else:
            b, m = idx // (K * (L + 1)), min(su[idx] - lo, hi - su[idx])
        dec[b] += 1
        near[b] += m < margin
    return dec, near


def verify_threads(mode, prob: Problem, threads=None, residual_out=False, trace_cap_per_request=4096):
    """verify() with the requests split into contiguous shares run on
    `threads` host threads (the oracle holds no global state, and ctypes
    releases the interpreter lock during each call).  Returns verify()'s
    outputs for the whole batch plus per-request 'decisions' and
    'near_margin' counts (trace_counts)."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    B = prob.B
    threads = max(1, min(threads or os.cpu_count() or 1, B)) if B else 1
    bounds = np.linspace(0, B, 4 * threads + 1).astype(int) if B else np.array([0, 0])
    shares = [(int(lo), int(hi)) for lo, hi in zip(bounds[:-1], bounds[1:]) if hi > lo]

    def run(share):
        lo, hi = share
        sub = prob.requests(lo, hi)
        out = verify(mode, sub, residual_out=residual_out, trace_cap=trace_cap_per_request * (hi - lo))
        out["decisions"], out["near_margin"] = trace_counts(sub, out["trace"])
        return out

    with ThreadPoolExecutor(max_workers=threads) as ex:
        parts = list(ex.map(run, shares))
    if any(p["rc"] != 0 for p in parts):
        raise RuntimeError("oracle verify failed")
    keys = ["accept_len", "accept_draft", "out_token", "accept_prob", "residual_mass", "margin", "req_status",
            "decisions", "near_margin"] + (["residual_out"] if residual_out else [])
    if not parts:
        empty = verify(mode, prob, residual_out=residual_out)
        empty["decisions"] = np.zeros(0, np.int64)
        empty["near_margin"] = np.zeros(0, np.int64)
        return empty
    out = {k: np.concatenate([p[k] for p in parts]) for k in keys}
    out["rc"] = 0
    return out


def sample_rows(logits, n_samples, u, temperature, V=None):
    """Draft-token sampling: n_samples inverse-CDF draws per row of
    softmax(logits / T).  logits [n_rows][stride] (f32, or bf16 as a CPU
    torch tensor or uint16 bits), u [n_rows][n_samples].  Returns a dict with
    tokens [n_rows][n_samples], margin [n_rows][n_samples], row_status
    [n_rows] and rc."""
    lg = _np(logits)
    n_rows, stride = lg.shape[0], lg.shape[1]
    V = stride if V is None else int(V)
    dtype = BF16 if lg.dtype in (np.uint16, np.int16) else F32
    uu = None if u is None else np.ascontiguousarray(_np(u), dtype=np.float64)
    out = {"tokens": np.zeros((n_rows, n_samples), np.int32),
           "margin": np.zeros((n_rows, n_samples), np.float64),
           "row_status": np.zeros(n_rows, np.int32)}
    rc = lib().sdvo_sample_rows(
        ctypes.c_int(n_rows), ctypes.c_int(V), ctypes.c_longlong(stride), ctypes.c_int(dtype),
        ctypes.c_double(float(temperature)), _ptr(lg), ctypes.c_int(n_samples), _ptr(uu),
        _ptr(out["tokens"]), _ptr(out["margin"]), _ptr(out["row_status"]))
    out["rc"] = rc
    return out


def lm_head_logits(hidden, lm_head):
    """The target model's LM head in double: hidden [..., d] and lm_head [V][d]
    as bf16 (CPU torch tensors or uint16 bits).  Returns float64 logits of
    shape hidden.shape[:-1] + (V,)."""
    h = _np(hidden)
    w = _np(lm_head)
    if h.dtype not in (np.uint16, np.int16) or w.dtype not in (np.uint16, np.int16):
        raise TypeError("the LM head takes bf16 inputs")
    d = h.shape[-1]
    if w.ndim != 2 or w.shape[1] != d:
        raise ValueError("lm_head must be [V][d] with the hidden size of hidden")
    lead = h.shape[:-1]
    M = int(np.prod(lead)) if lead else 1
    V = w.shape[0]
    out = np.zeros((M, V), np.float64)
    rc = lib().sdvo_lm_head_logits(ctypes.c_int(M), ctypes.c_int(V), ctypes.c_int(d),
                                   _ptr(np.ascontiguousarray(h)), _ptr(np.ascontiguousarray(w)),
                                   _ptr(out), ctypes.c_longlong(V))
    if rc != 0:
        raise RuntimeError(f"sdvo_lm_head_logits failed: {rc}")
    return out.reshape(tuple(lead) + (V,))


def exact_outcomes(mode, prob: Problem):
    """Exact P(tau, k*, token) of a one-request problem: array [L+1][K][V]."""
    assert prob.B == 1
    out = np.zeros((prob.L + 1, prob.K, prob.V), np.float64)
    s = prob.struct()
    rc = lib().sdvo_exact_outcomes(ctypes.c_int(MODE[mode]), ctypes.byref(s), _ptr(out))
    if rc != 0:
        raise RuntimeError(f"sdvo_exact_outcomes failed: {rc}")
    return out


def exact_accept_len(mode, prob: Problem):
    """Exact P(tau = i) of a one-request problem over its accept uniforms:
    array [L+1]."""
    assert prob.B == 1
    out = np.zeros(prob.L + 1, np.float64)
    s = prob.struct()
    rc = lib().sdvo_exact_accept_len(ctypes.c_int(MODE[mode]), ctypes.byref(s), _ptr(out))
    if rc != 0:
        raise RuntimeError(f"sdvo_exact_accept_len failed: {rc}")
    return out


def expected_accept_len(mode, prob: Problem, threads=None):
    """E[tau | drafts] of every request (exact over its accept uniforms),
    computed on host threads: array [B]."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    if prob.B == 0:
        return np.zeros(0)
    threads = max(1, min(threads or os.cpu_count() or 1, prob.B))
    with ThreadPoolExecutor(max_workers=threads) as ex:
        dists = list(ex.map(lambda b: exact_accept_len(mode, prob.request(b)), range(prob.B)))
    return np.array([float(np.dot(np.arange(d.size), d)) for d in dists])


def prefix_index(tokens, V):
    """Index of a prefix in the toy-model tables (all shorter prefixes first)."""
    off, pw = 0, 1
    for _ in range(len(tokens)):
        off += pw
        pw *= V
    num = 0
    for t in tokens:
        num = num * V + int(t)
    return off + num


def n_prefixes(n, V):
    """Number of prefixes of length 0..n."""
    return sum(V ** i for i in range(n + 1))


def exact_streams(mode, V, K, L, temperature, tgt_tab, dft_tab, q_tab):
    """Exact distribution of the emitted stream over all draft tuples.

    Tables hold one row per prefix of length 0..L (prefix_index order):
    f32 logits for target and draft, and the draft's sampling probabilities.
    Returns (stream_prob indexed by prefix_index over lengths 0..L+1,
    tau_prob[L+1]).
    """
    tgt = np.ascontiguousarray(tgt_tab, np.float32)
    dft = np.ascontiguousarray(dft_tab, np.float32)
    q = np.ascontiguousarray(q_tab, np.float64)
    sp = np.zeros(n_prefixes(L + 1, V), np.float64)
    tp = np.zeros(L + 1, np.float64)
    rc = lib().sdvo_exact_streams(ctypes.c_int(MODE[mode]), ctypes.c_int(V), ctypes.c_int(K),
                                  ctypes.c_int(L), ctypes.c_double(temperature),
                                  _ptr(tgt), _ptr(dft), _ptr(q), _ptr(sp), _ptr(tp))
    if rc != 0:
        raise RuntimeError(f"sdvo_exact_streams failed: {rc}")
    return sp, tp
