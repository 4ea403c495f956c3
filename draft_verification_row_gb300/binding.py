"""ctypes binding of libsdv.so (include/sdv.h).  Argument marshalling only."""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsdv.so")

MODES = {"token": 0, "greedy": 1, "block": 2, "multidraft": 3, "kseq": 4}
_ENTRY = {"token": "sdv_verify_token", "greedy": "sdv_verify_greedy",
          "block": "sdv_verify_block", "multidraft": "sdv_verify_multidraft", "kseq": "sdv_verify_kseq"}
SDV_F32, SDV_BF16 = 0, 1
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "CUDA error", 4: "timeout",
          5: "workspace"}
REQ_BAD_LENGTH, REQ_BAD_TOKEN, REQ_NONFINITE, DEV_TIMEOUT = 1, 2, 4, 8

_VERIFY_ARGTYPES = [
    ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_longlong, ctypes.c_int,
    ctypes.c_float,
    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
    ctypes.c_void_p,
    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
]

EXPORTS = list(_ENTRY.values()) + ["sdv_workspace_bytes", "sdv_status_string", "sdv_launch_shape",
                                   "sdv_set_profile_events", "sdv_sample_rows", "sdv_copy_read_rows",
                                   "sdv_read_rows_bytes", "sdv_gather_read_rows", "sdv_verify_greedy_lm_head",
                                   "sdv_lm_head_workspace_bytes", "sdv_lm_head_logits", "sdv_gather_inner_rows",
                                   "sdv_verify_leaves_apart", "sdv_lm_head_trie_logits", "sdv_verify_residual",
                                   "sdv_verify_multidraft_static", "sdv_testing_set_wait_limit",
                                   "sdv_testing_verify_without_roots", "sdv_testing_set_lm_head_single_cta"]


class SDVError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"{what}: {STATUS.get(code, code)} ({code})")
        self.code = code


_lib = None


def lib(path: str = LIB_PATH):
    """Load libsdv.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    h = ctypes.CDLL(path)
    for name in _ENTRY.values():
        fn = getattr(h, name)
        fn.restype = ctypes.c_int
        fn.argtypes = _VERIFY_ARGTYPES
    h.sdv_workspace_bytes.restype = ctypes.c_size_t
    h.sdv_workspace_bytes.argtypes = [ctypes.c_int] * 5
    h.sdv_status_string.restype = ctypes.c_char_p
    h.sdv_status_string.argtypes = [ctypes.c_int]
    h.sdv_launch_shape.restype = ctypes.c_int
    h.sdv_launch_shape.argtypes = [ctypes.c_int, ctypes.c_int] + [ctypes.POINTER(ctypes.c_int)] * 3
    h.sdv_set_profile_events.restype = ctypes.c_int
    h.sdv_set_profile_events.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    h.sdv_sample_rows.restype = ctypes.c_int
    h.sdv_sample_rows.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_longlong, ctypes.c_int, ctypes.c_float,
                                  ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                  ctypes.c_void_p, ctypes.c_void_p]
    h.sdv_copy_read_rows.restype = ctypes.c_int
    h.sdv_copy_read_rows.argtypes = ([ctypes.c_int] * 4 + [ctypes.c_longlong, ctypes.c_int] + [ctypes.c_void_p] * 7
                                     + [ctypes.POINTER(ctypes.c_longlong)])
    h.sdv_gather_read_rows.restype = ctypes.c_int
    h.sdv_gather_read_rows.argtypes = [ctypes.c_int] * 4 + [ctypes.c_longlong, ctypes.c_int] + [ctypes.c_void_p] * 7
    h.sdv_verify_greedy_lm_head.restype = ctypes.c_int
    h.sdv_verify_greedy_lm_head.argtypes = ([ctypes.c_int] * 5 + [ctypes.c_void_p] * 10 + [ctypes.c_size_t]
                                            + [ctypes.c_void_p])
    h.sdv_lm_head_workspace_bytes.restype = ctypes.c_size_t
    h.sdv_lm_head_workspace_bytes.argtypes = [ctypes.c_int] * 5
    h.sdv_lm_head_trie_logits.restype = ctypes.c_int
    h.sdv_lm_head_trie_logits.argtypes = ([ctypes.c_int] * 5 + [ctypes.c_void_p] * 5 + [ctypes.c_longlong]
                                          + [ctypes.c_void_p] * 2 + [ctypes.c_size_t, ctypes.c_void_p])
    h.sdv_lm_head_logits.restype = ctypes.c_int
    h.sdv_lm_head_logits.argtypes = ([ctypes.c_int] * 3 + [ctypes.c_void_p] * 3 + [ctypes.c_longlong]
                                     + [ctypes.c_void_p] * 2)
    h.sdv_gather_inner_rows.restype = ctypes.c_int
    h.sdv_gather_inner_rows.argtypes = h.sdv_gather_read_rows.argtypes
    h.sdv_verify_leaves_apart.restype = ctypes.c_int
    h.sdv_verify_leaves_apart.argtypes = [ctypes.c_int] + _VERIFY_ARGTYPES + [ctypes.c_void_p]
    h.sdv_verify_residual.restype = ctypes.c_int
    h.sdv_verify_residual.argtypes = [ctypes.c_int] + _VERIFY_ARGTYPES + [ctypes.c_void_p]
    h.sdv_testing_set_wait_limit.restype = ctypes.c_int
    h.sdv_testing_set_wait_limit.argtypes = [ctypes.c_ulonglong]
    h.sdv_testing_set_lm_head_single_cta.restype = ctypes.c_int
    h.sdv_testing_set_lm_head_single_cta.argtypes = [ctypes.c_int]
    h.sdv_testing_verify_without_roots.restype = ctypes.c_int
    h.sdv_testing_verify_without_roots.argtypes = [ctypes.c_int] + _VERIFY_ARGTYPES
    h.sdv_read_rows_bytes.restype = ctypes.c_int
    h.sdv_read_rows_bytes.argtypes = ([ctypes.c_int] * 4 + [ctypes.c_longlong, ctypes.c_int] + [ctypes.c_void_p] * 2
                                      + [ctypes.POINTER(ctypes.c_longlong)])
    _lib = h
    return h


def workspace_bytes(mode, B, K, L, V):
    return int(lib().sdv_workspace_bytes(MODES[mode], B, K, L, V))


def launch_shape(V, dtype="bf16"):
    c, t, s = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    rc = lib().sdv_launch_shape(V, SDV_BF16 if dtype == "bf16" else SDV_F32,
                                ctypes.byref(c), ctypes.byref(t), ctypes.byref(s))
    if rc:
        raise SDVError(rc, "sdv_launch_shape")
    return {"ctas_per_sm": c.value, "threads": t.value, "smem_bytes": s.value}


def set_profile_events(start=None, stop=None):
    """Record two torch.cuda.Events around the vocabulary-row kernels of each
    later call from this thread (None, None turns it off).  The events must
    have been recorded once so that they exist."""
    hs = None if start is None else ctypes.c_void_p(start.cuda_event)
    he = None if stop is None else ctypes.c_void_p(stop.cuda_event)
    rc = lib().sdv_set_profile_events(hs, he)
    if rc:
        raise SDVError(rc, "sdv_set_profile_events")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return SDV_BF16
    if t.dtype == torch.float32:
        return SDV_F32
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


class Outputs:
    """Preallocated outputs (and workspace) for repeated calls of one shape."""

    def __init__(self, mode, B, K, L, V, device, accept_prob=True, residual_mass=True, residual_out=False):
        self.residual_out = torch.empty((B, V), dtype=torch.float32, device=device) if residual_out else None
        self.accept_len = torch.empty(B, dtype=torch.int32, device=device)
        self.accept_draft = torch.empty(B, dtype=torch.int32, device=device)
        self.out_token = torch.empty(B, dtype=torch.int32, device=device)
        self.accept_prob = torch.empty((B, K, L), dtype=torch.float32, device=device) if accept_prob else None
        self.residual_mass = torch.empty(B, dtype=torch.float32, device=device) if residual_mass else None
        self.device_status = torch.empty(1, dtype=torch.int32, device=device)
        nbytes = max(workspace_bytes(mode, B, K, L, V), 256)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)

    def as_dict(self):
        d = {k: getattr(self, k) for k in ("accept_len", "accept_draft", "out_token", "accept_prob",
                                           "residual_mass", "device_status")}
        if self.residual_out is not None:
            d["residual_out"] = self.residual_out
        return d


def verify(mode, target, draft, tokens, lengths, accept_u, sample_u, temperature, *, V=None,
           out: Outputs = None, stream=None, accept_prob=True, residual_mass=True, leaf_target=None,
           residual_out=False):
    """Run one verification call on the current CUDA stream.

    target [B][K][L+1][stride], draft [B][K][L][stride] (float32 or bfloat16),
    tokens [B][K][L] int32, lengths [B] int32 or None, accept_u [B][K][L],
    sample_u [B][K][L+1] float32.  Returns a dict of output tensors; the call
    is asynchronous (read them after a synchronize).  leaf_target: a tensor of
    target's shape and dtype (e.g. pinned host memory) the leaves' rows are
    read from instead (sdv_verify_leaves_apart).  residual_out: also return
    [B][V] float32 rows, the normalised distribution each correction was
    drawn from (sdv_verify_residual).
    """
    if mode not in _ENTRY:
        raise ValueError(f"unknown mode {mode!r}")
    h = lib()
    if target.dim() != 4:
        raise ValueError("target must be [B][K][L+1][stride]")
    B, K, Lp1, stride = target.shape
    L = Lp1 - 1
    V = stride if V is None else int(V)
    for name, t in (("target", target), ("draft", draft)):
        if t is not None and (not t.is_contiguous() or not t.is_cuda):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if draft is not None and draft.dtype != target.dtype:
        raise TypeError("target and draft logits must have the same dtype")
    for name, t, dt in (("tokens", tokens, torch.int32), ("lengths", lengths, torch.int32),
                        ("accept_u", accept_u, torch.float32), ("sample_u", sample_u, torch.float32)):
        if t is not None and (t.dtype != dt or not t.is_contiguous() or not t.is_cuda):
            raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor")
    if out is None:
        out = Outputs(mode, B, K, L, V, target.device, accept_prob, residual_mass, residual_out)
    if residual_out and (out.residual_out is None or tuple(out.residual_out.shape) != (B, V)):
        raise ValueError("residual_out needs Outputs holding a [B][V] residual_out tensor")
    if residual_out and leaf_target is not None:
        raise ValueError("residual_out and leaf_target cannot be combined")
    if stream is None:
        stream = torch.cuda.current_stream(target.device)
    args = (B, K, L, V, stride, _dtype_code(target), float(temperature),
            _ptr(target), _ptr(draft), _ptr(tokens), _ptr(lengths), _ptr(accept_u), _ptr(sample_u),
            _ptr(out.accept_len), _ptr(out.accept_draft), _ptr(out.out_token), _ptr(out.accept_prob),
            _ptr(out.residual_mass), _ptr(out.device_status), _ptr(out.workspace),
            out.workspace.numel(), ctypes.c_void_p(stream.cuda_stream))
    if residual_out:
        rc = h.sdv_verify_residual(MODES[mode], *args, _ptr(out.residual_out))
        if rc != 0:
            raise SDVError(rc, "sdv_verify_residual")
        return out.as_dict()
    if leaf_target is None:
        rc = getattr(h, _ENTRY[mode])(*args)
    else:
        if leaf_target.shape != target.shape or leaf_target.dtype != target.dtype or not leaf_target.is_contiguous():
            raise ValueError("leaf_target must be contiguous, with target's shape and dtype")
        rc = h.sdv_verify_leaves_apart(MODES[mode], *args, _ptr(leaf_target))
    if rc != 0:
        raise SDVError(rc, _ENTRY[mode] if leaf_target is None else "sdv_verify_leaves_apart")
    return out.as_dict()


def verify_token(*args, **kw):
    return verify("token", *args, **kw)


def verify_greedy(*args, **kw):
    return verify("greedy", *args, **kw)


def verify_block(*args, **kw):
    return verify("block", *args, **kw)


def verify_multidraft(*args, **kw):
    return verify("multidraft", *args, **kw)


def verify_kseq(*args, **kw):
    return verify("kseq", *args, **kw)


def sample_rows(logits, n_samples, u, temperature, *, V=None, tokens=None, device_status=None, stream=None):
    """Draft-token sampling: n_samples inverse-CDF draws per row of
    softmax(logits / T).

    logits [n_rows][width] (float32 or bfloat16, CUDA; each row contiguous,
    rows evenly spaced by logits.stride(0), e.g. one depth's rows of a
    [B][K][L][stride] draft tensor), u [n_rows][n_samples] float32 (may be
    None when T == 0).  Returns (tokens [n_rows][n_samples] int32,
    device_status [1] int32); the call is asynchronous.
    """
    h = lib()
    if logits.dim() != 2 or not logits.is_cuda or (logits.shape[0] > 1 and logits.stride(1) != 1):
        raise ValueError("logits must be a CUDA [n_rows][width] tensor with contiguous rows")
    n_rows, width = logits.shape
    stride = logits.stride(0) if n_rows > 1 else width
    V = width if V is None else int(V)
    if u is not None and (u.dtype != torch.float32 or not u.is_cuda or not u.is_contiguous()
                          or tuple(u.shape) != (n_rows, n_samples)):
        raise ValueError("u must be a contiguous CUDA float32 [n_rows][n_samples] tensor")
    if tokens is None:
        tokens = torch.empty((n_rows, n_samples), dtype=torch.int32, device=logits.device)
    if device_status is None:
        device_status = torch.empty(1, dtype=torch.int32, device=logits.device)
    if stream is None:
        stream = torch.cuda.current_stream(logits.device)
    rc = h.sdv_sample_rows(n_rows, V, stride, _dtype_code(logits), float(temperature), _ptr(logits),
                           int(n_samples), _ptr(u), _ptr(tokens), _ptr(device_status),
                           ctypes.c_void_p(stream.cuda_stream))
    if rc != 0:
        raise SDVError(rc, "sdv_sample_rows")
    return tokens, device_status



def _bf16_rows(name, t, d=None):
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA bfloat16 tensor")
    if d is not None and t.shape[-1] != d:
        raise ValueError(f"{name} must have the hidden size {d} as its last dimension")


class LmHeadOutputs:
    """Preallocated outputs and workspace of verify_greedy_lm_head for one shape."""

    def __init__(self, B, K, L, V, d, device, accept_prob=True):
        self.accept_len = torch.empty(B, dtype=torch.int32, device=device)
        self.accept_draft = torch.empty(B, dtype=torch.int32, device=device)
        self.out_token = torch.empty(B, dtype=torch.int32, device=device)
        self.accept_prob = torch.empty((B, K, L), dtype=torch.float32, device=device) if accept_prob else None
        self.device_status = torch.empty(1, dtype=torch.int32, device=device)
        nbytes = max(lib().sdv_lm_head_workspace_bytes(B, K, L, V, d), 256)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)

    def as_dict(self):
        return {k: getattr(self, k) for k in ("accept_len", "accept_draft", "out_token", "accept_prob",
                                              "device_status")}


def lm_head_workspace_bytes(B, K, L, V, d):
    return lib().sdv_lm_head_workspace_bytes(B, K, L, V, d)


def verify_greedy_lm_head(hidden, lm_head, tokens, lengths, *, out: LmHeadOutputs = None, stream=None,
                          accept_prob=True):
    """Greedy verification fused into the target model's LM head.

    hidden [B][K][L+1][d] bfloat16 (the target model's final hidden state of
    every draft position), lm_head [V][d] bfloat16, tokens [B][K][L] int32,
    lengths [B] int32 or None.  Returns a dict of output tensors
    (asynchronous, like verify)."""
    h = lib()
    if hidden.dim() != 4 or lm_head.dim() != 2:
        raise ValueError("hidden must be [B][K][L+1][d] and lm_head [V][d]")
    B, K, Lp1, d = hidden.shape
    L, V = Lp1 - 1, lm_head.shape[0]
    _bf16_rows("hidden", hidden)
    _bf16_rows("lm_head", lm_head, d)
    for name, t in (("tokens", tokens), ("lengths", lengths)):
        if t is not None and (t.dtype != torch.int32 or not t.is_contiguous() or not t.is_cuda):
            raise ValueError(f"{name} must be a contiguous CUDA int32 tensor")
    if out is None:
        out = LmHeadOutputs(B, K, L, V, d, hidden.device, accept_prob)
    if stream is None:
        stream = torch.cuda.current_stream(hidden.device)
    rc = h.sdv_verify_greedy_lm_head(B, K, L, V, d, _ptr(hidden), _ptr(lm_head), _ptr(tokens), _ptr(lengths),
                                     _ptr(out.accept_len), _ptr(out.accept_draft), _ptr(out.out_token),
                                     _ptr(out.accept_prob), _ptr(out.device_status), _ptr(out.workspace),
                                     out.workspace.numel(), ctypes.c_void_p(stream.cuda_stream))
    if rc != 0:
        raise SDVError(rc, "sdv_verify_greedy_lm_head")
    return out.as_dict()


def lm_head_trie_logits(hidden, lm_head, tokens, lengths, *, target=None, workspace=None, device_status=None,
                        stream=None):
    """The target logits of every trie node (leaves included), computed once
    by the LM head and written in bf16 into target [B][K][L+1][stride] (a
    new NaN-filled tensor with stride V rounded up to 8 when None): the rows
    the sampling rules read (sdv_lm_head_trie_logits).  Returns (target,
    device_status); asynchronous."""
    h = lib()
    if hidden.dim() != 4 or lm_head.dim() != 2:
        raise ValueError("hidden must be [B][K][L+1][d] and lm_head [V][d]")
    B, K, Lp1, d = hidden.shape
    L, V = Lp1 - 1, lm_head.shape[0]
    _bf16_rows("hidden", hidden)
    _bf16_rows("lm_head", lm_head, d)
    if target is None:
        target = torch.full((B, K, Lp1, (V + 7) // 8 * 8), float("nan"), dtype=torch.bfloat16, device=hidden.device)
    if target.dtype != torch.bfloat16 or not target.is_contiguous() or tuple(target.shape[:3]) != (B, K, Lp1):
        raise ValueError("target must be a contiguous bfloat16 [B][K][L+1][stride] tensor")
    if workspace is None:
        workspace = torch.empty(max(h.sdv_lm_head_workspace_bytes(B, K, L, V, d), 256), dtype=torch.uint8,
                                device=hidden.device)
    if device_status is None:
        device_status = torch.empty(1, dtype=torch.int32, device=hidden.device)
    if stream is None:
        stream = torch.cuda.current_stream(hidden.device)
    rc = h.sdv_lm_head_trie_logits(B, K, L, V, d, _ptr(hidden), _ptr(lm_head), _ptr(tokens), _ptr(lengths),
                                   _ptr(target), target.shape[3], _ptr(device_status), _ptr(workspace),
                                   workspace.numel(), ctypes.c_void_p(stream.cuda_stream))
    if rc != 0:
        raise SDVError(rc, "sdv_lm_head_trie_logits")
    return target, device_status


def lm_head_logits(hidden, lm_head, *, logits=None, device_status=None, stream=None):
    """The target model's LM head alone: fp32 logits [M][V] of hidden [M][d]
    and lm_head [V][d] (bfloat16).  logits may be a preallocated float32
    [M][>= V] tensor with contiguous rows (row stride a multiple of 4).
    Returns (logits, device_status); asynchronous."""
    h = lib()
    if hidden.dim() != 2 or lm_head.dim() != 2:
        raise ValueError("hidden must be [M][d] and lm_head [V][d]")
    M, d = hidden.shape
    V = lm_head.shape[0]
    _bf16_rows("hidden", hidden)
    _bf16_rows("lm_head", lm_head, d)
    if logits is None:
        logits = torch.empty((M, V), dtype=torch.float32, device=hidden.device)
    if (logits.dtype != torch.float32 or not logits.is_cuda or logits.shape[0] != M or logits.shape[1] < V
            or logits.stride(1) != 1):
        raise ValueError("logits must be a CUDA float32 [M][>= V] tensor with contiguous rows")
    if device_status is None:
        device_status = torch.empty(1, dtype=torch.int32, device=hidden.device)
    if stream is None:
        stream = torch.cuda.current_stream(hidden.device)
    rc = h.sdv_lm_head_logits(M, V, d, _ptr(hidden), _ptr(lm_head), _ptr(logits), logits.stride(0),
                              _ptr(device_status), ctypes.c_void_p(stream.cuda_stream))
    if rc != 0:
        raise SDVError(rc, "sdv_lm_head_logits")
    return logits, device_status


def _host_i32(t):
    if t is None:
        return None
    if t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous():
        raise ValueError("tokens and lengths must be contiguous int32 host tensors")
    return t


def read_rows_bytes(tokens, lengths, V, row_stride, dtype):
    """Bytes of the rows verification reads (sdv_read_rows_bytes); tokens
    [B][K][L] and lengths [B] are int32 host tensors."""
    B, K, L = tokens.shape
    out = ctypes.c_longlong(0)
    rc = lib().sdv_read_rows_bytes(B, K, L, int(V), int(row_stride), SDV_BF16 if dtype == torch.bfloat16 else SDV_F32,
                                   _ptr(_host_i32(tokens)), _ptr(_host_i32(lengths)), ctypes.byref(out))
    if rc != 0:
        raise SDVError(rc, "sdv_read_rows_bytes")
    return out.value


def copy_read_rows(host_target, host_draft, tokens, lengths, target, draft, *, V=None, stream=None):
    """Queue host-to-device copies of the rows verification reads
    (sdv_copy_read_rows).  host_target / host_draft: full host tensors
    (pinned); tokens / lengths: int32 host tensors; target / draft: device
    tensors of the same shapes.  Returns the bytes queued."""
    B, K, Lp1, stride = host_target.shape
    V = stride if V is None else int(V)
    if stream is None:
        stream = torch.cuda.current_stream(target.device)
    out = ctypes.c_longlong(0)
    rc = lib().sdv_copy_read_rows(B, K, Lp1 - 1, V, stride, _dtype_code(host_target), _ptr(host_target),
                                  _ptr(host_draft), _ptr(_host_i32(tokens)), _ptr(_host_i32(lengths)),
                                  _ptr(target), _ptr(draft), ctypes.c_void_p(stream.cuda_stream), ctypes.byref(out))
    if rc != 0:
        raise SDVError(rc, "sdv_copy_read_rows")
    return out.value


def gather_read_rows(host_target, host_draft, tokens, lengths, target, draft, *, V=None, stream=None,
                     leaves=True):
    """Gather the rows verification reads from pinned, device-mapped host
    tensors into device tensors with one kernel (sdv_gather_read_rows);
    tokens / lengths are the device tensors the verification call takes.
    leaves=False leaves out the leaves' target rows (sdv_gather_inner_rows):
    verify(..., leaf_target=host_target) then reads the few it needs from
    the host tensor."""
    B, K, Lp1, stride = host_target.shape
    V = stride if V is None else int(V)
    if stream is None:
        stream = torch.cuda.current_stream(target.device)
    name = "sdv_gather_read_rows" if leaves else "sdv_gather_inner_rows"
    rc = getattr(lib(), name)(B, K, Lp1 - 1, V, stride, _dtype_code(host_target), _ptr(host_target),
                              _ptr(host_draft), _ptr(tokens), _ptr(lengths), _ptr(target), _ptr(draft),
                              ctypes.c_void_p(stream.cuda_stream))
    if rc != 0:
        raise SDVError(rc, name)
