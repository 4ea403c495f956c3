"""Batched speculative-decoding verification on GB300 (sm_103a), and the
draft-token sampling step before it.

A thin ctypes binding of the C-ABI in include/sdv.h (libsdv.so, built
in-tree by ``draft_verification_row_gb300.build``).  Every step of the
verification runs in the library's CUDA kernels; this module only checks
tensor shapes, takes pointers and the current stream, and allocates the
workspace and outputs with torch.  There is no CPU fallback: without the
compiled library every call raises.
"""
from .binding import (  # noqa: F401
    MODES,
    SDVError,
    copy_read_rows,
    gather_read_rows,
    launch_shape,
    lib,
    lm_head_logits,
    lm_head_trie_logits,
    lm_head_workspace_bytes,
    read_rows_bytes,
    sample_rows,
    set_profile_events,
    verify,
    verify_block,
    verify_greedy,
    verify_greedy_lm_head,
    verify_kseq,
    verify_multidraft,
    verify_token,
    workspace_bytes,
)
