"""The Python binding rejects malformed tensors before calling the library
(no GPU needed: every case fails in the argument checks)."""
import pytest
import torch

import draft_verification_row_gb300 as sdv


def _verify_args(B=2, K=2, L=2, V=16, dtype=torch.float32, dev="cpu"):
    t = torch.zeros((B, K, L + 1, V), dtype=dtype, device=dev)
    d = torch.zeros((B, K, L, V), dtype=dtype, device=dev)
    tok = torch.zeros((B, K, L), dtype=torch.int32, device=dev)
    ln = torch.full((B,), L, dtype=torch.int32, device=dev)
    au = torch.zeros((B, K, L), device=dev)
    su = torch.zeros((B, K, L + 1), device=dev)
    return t, d, tok, ln, au, su


def test_unknown_mode():
    with pytest.raises(ValueError, match="unknown mode"):
        sdv.verify("nope", *_verify_args(), 1.0)


def test_host_tensors_are_refused():
    with pytest.raises(ValueError, match="CUDA"):
        sdv.verify("token", *_verify_args(), 1.0)


def test_target_must_be_four_dimensional():
    t, d, tok, ln, au, su = _verify_args()
    with pytest.raises(ValueError, match="target"):
        sdv.verify("token", t[0], d, tok, ln, au, su, 1.0)


def test_lm_head_inputs_must_be_bf16_and_shaped():
    h = torch.zeros((2, 2, 3, 16), dtype=torch.float32)
    w = torch.zeros((32, 16), dtype=torch.float32)
    tok = torch.zeros((2, 2, 2), dtype=torch.int32)
    with pytest.raises(ValueError, match="bfloat16"):
        sdv.verify_greedy_lm_head(h, w, tok, None)
    with pytest.raises(ValueError, match="bfloat16"):
        sdv.lm_head_trie_logits(h, w, tok, None)
    with pytest.raises(ValueError):
        sdv.lm_head_logits(h[0, 0], w)
    with pytest.raises(ValueError, match=r"\[V\]\[d\]|\[M\]\[d\]"):
        sdv.lm_head_logits(h, w)


def test_lm_head_host_tensors_are_refused():
    h = torch.zeros((4, 16), dtype=torch.bfloat16)
    w = torch.zeros((32, 16), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        sdv.lm_head_logits(h, w)
