"""The C-ABI library on the host: it loads, exports what include/sdv.h
declares, and rejects invalid arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from draft_verification_row_gb300 import build
    build.build()
    import draft_verification_row_gb300 as sdv
    return sdv.lib()


def _declared():
    inc = os.path.join(ROOT, "include")
    src = "".join(open(os.path.join(inc, f)).read() for f in sorted(os.listdir(inc)) if f.endswith(".h"))
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sdv_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert "sdv_verify_multidraft" in names and len(names) >= 7
    for n in names:
        assert hasattr(lib, n), n


def test_workspace_bytes(lib):
    import draft_verification_row_gb300 as sdv
    assert sdv.workspace_bytes("multidraft", 256, 8, 8, 151936) > 256 * 8 * 9 * 24
    assert sdv.workspace_bytes("token", 0, 1, 0, 1) >= 0
    assert lib.sdv_workspace_bytes(2, 4, 2, 4, 100) == 0      # block needs K = 1
    assert lib.sdv_workspace_bytes(0, 4, 0, 4, 100) == 0      # K = 0
    assert lib.sdv_workspace_bytes(0, 4, 1, 17, 100) == 0     # L > 16
    assert lib.sdv_workspace_bytes(0, 4, 1, 4, 262145) == 0   # V > max
    assert lib.sdv_workspace_bytes(7, 4, 1, 4, 100) == 0      # unknown mode


@pytest.mark.parametrize("V,dtype", [(1024, "f32"), (32000, "bf16"), (151936, "bf16"), (262144, "f32")])
def test_launch_shape(lib, V, dtype):
    import draft_verification_row_gb300 as sdv
    s = sdv.launch_shape(V, dtype)
    assert s["ctas_per_sm"] >= 1
    assert s["ctas_per_sm"] * (s["smem_bytes"] + 1024) <= 228 * 1024  # fits an SM's shared memory
    assert s["threads"] % 32 == 0 and s["ctas_per_sm"] * s["threads"] <= 2048
    with pytest.raises(sdv.SDVError):
        sdv.launch_shape(262145, dtype)


def test_status_strings(lib):
    assert lib.sdv_status_string(0) == b"ok"
    assert b"workspace" in lib.sdv_status_string(5)


def _call(lib, name, **over):
    a = dict(B=2, K=1, L=2, V=16, stride=16, dtype=0, T=1.0)
    a.update(over)
    fn = getattr(lib, name)
    return fn(a["B"], a["K"], a["L"], a["V"], a["stride"], a["dtype"], a["T"],
              None, None, None, None, None, None, None, None, None, None, None, None, None, 0, None)


@pytest.mark.parametrize("over", [dict(K=0), dict(K=17), dict(L=-1), dict(L=17), dict(V=0),
                                  dict(V=262145, stride=262152), dict(stride=12), dict(stride=8),
                                  dict(dtype=2), dict(T=-1.0), dict(T=float("nan")), dict(T=float("inf")),
                                  dict(B=-1)])
def test_invalid_sizes_rejected_without_gpu(lib, over):
    assert _call(lib, "sdv_verify_token", **over) == 1


def test_block_rejects_multiple_drafts(lib):
    assert _call(lib, "sdv_verify_block", K=2) == 1


def test_empty_batch_is_a_no_op(lib):
    assert _call(lib, "sdv_verify_multidraft", B=0) == 0


def test_package_fails_loudly_without_library(tmp_path):
    from draft_verification_row_gb300 import binding
    saved = binding._lib
    binding._lib = None
    try:
        with pytest.raises(ImportError):
            binding.lib(str(tmp_path / "missing.so"))
    finally:
        binding._lib = saved


def test_read_rows_bytes_match_the_trie(lib):
    """The rows verification reads, counted by the library on the host: per
    request and draft, target rows from the first depth the draft owns to
    L_b and draft rows to L_b - 1 (the trie rows of the bench's count: one
    pair per inner node plus a target row per leaf)."""
    import bench
    import draft_verification_row_gb300 as sdv
    from draft_verification_row_gb300 import workloads as W
    batch = W.make("mixed-B256-K8-L8-V151936-bf16", "cpu", B=12, V=997)
    inner, leaves = bench.trie_nodes(batch.tokens, batch.lengths, batch.K)
    got = sdv.read_rows_bytes(batch.tokens, batch.lengths, batch.V, batch.stride, batch.target.dtype)
    assert got == (2 * inner + leaves) * batch.stride * 2
    # a request with an out-of-range length reads nothing
    lengths = batch.lengths.clone()
    lengths[0] = batch.L + 1
    inner0, leaves0 = bench.trie_nodes(batch.tokens[1:], batch.lengths[1:], batch.K)
    assert sdv.read_rows_bytes(batch.tokens, lengths, batch.V, batch.stride, batch.target.dtype) == \
        (2 * inner0 + leaves0) * batch.stride * 2


def test_lm_head_workspace_bytes(lib):
    n = 256 * 8 * 9
    ws = lib.sdv_lm_head_workspace_bytes(256, 8, 8, 151936, 4096)
    # the verification workspace, the nodes' hidden rows, their keys and map
    assert ws >= lib.sdv_workspace_bytes(1, 256, 8, 8, 151936) + n * (4096 * 2 + 8 + 4)
    for bad in [(1, 1, 1, 16, 0), (1, 1, 1, 16, 12), (1, 1, 1, 16, 1 << 17), (1, 0, 1, 16, 64),
                (1, 1, 17, 16, 64), (1, 1, 1, 262145, 64), (-1, 1, 1, 16, 64)]:
        assert lib.sdv_lm_head_workspace_bytes(*bad) == 0, bad


@pytest.mark.parametrize("over", [dict(d=0), dict(d=12), dict(d=1 << 17), dict(K=0), dict(K=17), dict(L=17),
                                  dict(V=0), dict(V=262145), dict(B=-1)])
def test_lm_head_invalid_sizes_rejected_without_gpu(lib, over):
    a = dict(B=2, K=1, L=2, V=16, d=64)
    a.update(over)
    assert lib.sdv_verify_greedy_lm_head(a["B"], a["K"], a["L"], a["V"], a["d"], *([None] * 10), 0, None) == 1


@pytest.mark.parametrize("over", [dict(M=-1), dict(V=0), dict(V=262145, stride=262148), dict(d=4), dict(d=20),
                                  dict(stride=12), dict(stride=18)])
def test_lm_head_logits_invalid_rejected_without_gpu(lib, over):
    a = dict(M=2, V=16, d=64, stride=16)
    a.update(over)
    assert lib.sdv_lm_head_logits(a["M"], a["V"], a["d"], None, None, None, a["stride"], None, None) == 1


def test_lm_head_empty_is_a_no_op(lib):
    assert lib.sdv_verify_greedy_lm_head(0, 2, 2, 16, 64, *([None] * 10), 0, None) == 0
    assert lib.sdv_lm_head_logits(0, 16, 64, None, None, None, 16, None, None) == 0


@pytest.mark.parametrize("mode", [-1, 5])
def test_leaves_apart_rejects_unknown_modes_without_gpu(lib, mode):
    args = [2, 1, 2, 16, 16, 0, 1.0] + [None] * 13 + [0, None]
    assert lib.sdv_verify_leaves_apart(mode, *args, None) == 1


def test_leaves_apart_checks_sizes_without_gpu(lib):
    args = [2, 0, 2, 16, 16, 0, 1.0] + [None] * 13 + [0, None]  # K = 0
    assert lib.sdv_verify_leaves_apart(3, *args, None) == 1
    args = [0, 1, 2, 16, 16, 0, 1.0] + [None] * 13 + [0, None]  # B = 0: nothing to do
    assert lib.sdv_verify_leaves_apart(3, *args, None) == 0


def test_gather_inner_rows_rejects_bad_sizes_without_gpu(lib):
    f = lib.sdv_gather_inner_rows
    assert f(2, 0, 2, 16, 16, 1, None, None, None, None, None, None, None) == 1   # K = 0
    assert f(2, 1, 2, 16, 12, 1, None, None, None, None, None, None, None) == 1   # stride < V
    assert f(0, 1, 2, 16, 16, 1, None, None, None, None, None, None, None) == 0   # B = 0


@pytest.mark.parametrize("over", [dict(d=12), dict(K=0), dict(L=17), dict(V=0), dict(stride=12), dict(stride=20),
                                  dict(B=-1)])
def test_trie_logits_invalid_sizes_rejected_without_gpu(lib, over):
    a = dict(B=2, K=1, L=2, V=16, d=64, stride=16)
    a.update(over)
    assert lib.sdv_lm_head_trie_logits(a["B"], a["K"], a["L"], a["V"], a["d"], None, None, None, None, None,
                                       a["stride"], None, None, 0, None) == 1


def test_trie_logits_empty_batch_is_a_no_op(lib):
    assert lib.sdv_lm_head_trie_logits(0, 2, 2, 16, 64, None, None, None, None, None, 16, None, None, 0, None) == 0
