"""One-GPU emulation of batch-parallel speculative decoding (PSD).

The MineDraft pages (section 2, "two batches") describe the method: requests
are kept in two batches, and while the target model verifies one batch, the
draft model drafts the other; at the end of each speculative step the two
swap roles, so that drafting is hidden behind verification.  The pages run
the draft model on a GPU of its own.  Here both phases share one GPU, on two
CUDA streams, and the phases are stand-ins built from this library's kernels:

  draft phase    L launches of sdv_sample_rows, one per depth: each draft's
                 next token drawn from its draft row at that depth (the row
                 a draft model would have produced; synthetic here), written
                 into the batch's draft tokens;
  verify phase   one SpecTr-GBV verification call over the batch.

No draft or target model runs (there are no weights), so the emulation
measures how much of one phase's kernel time the other hides on a shared
GPU, not the pages' end-to-end latency.  The batch manager keeps two fixed
halves of a batch; requests never finish or move.

Every tensor is created up front; a step only launches kernels and joins
the two streams at its end.
"""
from dataclasses import dataclass
from typing import List, Optional

import torch

from . import binding


def roles(step: int):
    """(verifying batch, drafting batch) at a step: batch 0 verifies first."""
    return step % 2, 1 - step % 2


def hidden_fraction(t_draft: float, t_verify: float, t_seq: float, t_psd: float) -> float:
    """Share of the shorter phase hidden by the overlap: 0 when a PSD step
    takes as long as the two phases one after the other, 1 when it takes as
    long as the longer phase alone."""
    shorter = min(t_draft, t_verify)
    return 0.0 if shorter <= 0 else (t_seq - t_psd) / shorter


@dataclass
class Half:
    """One batch of requests: views of a workload batch's tensors plus the
    buffers its two phases write."""
    target: torch.Tensor      # [B][K][L+1][stride]
    draft: torch.Tensor       # [B][K][L][stride]
    tokens: torch.Tensor      # [B][K][L] int32, written by the draft phase
    lengths: torch.Tensor
    accept_u: torch.Tensor
    sample_u: torch.Tensor
    draft_u: torch.Tensor     # [steps][L][B*K] float32: the draft phase's uniforms
    tok: torch.Tensor         # [L][B*K][1] int32: sampled tokens by depth
    status: torch.Tensor      # [1] int32: sampling status
    out: binding.Outputs


class PsdEmulator:
    """Two halves of a workload batch alternating draft and verify phases.

    batch: a workloads.Batch (B even); steps: how many steps the prepared
    uniforms cover (a step index wraps around beyond that)."""

    def __init__(self, batch, steps: int = 8, seed: int = 0):
        if batch.B % 2 or batch.B == 0 or batch.L == 0:
            raise ValueError("PSD needs an even, non-empty batch and L >= 1")
        self.B, self.K, self.L, self.V = batch.B // 2, batch.K, batch.L, batch.V
        self.T = batch.temperature
        self.steps = steps
        dev = batch.target.device
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        self.halves: List[Half] = []
        for h in range(2):
            sl = slice(h * self.B, (h + 1) * self.B)
            n = self.B * self.K
            self.halves.append(Half(
                target=batch.target[sl], draft=batch.draft[sl], tokens=batch.tokens[sl].clone(),
                lengths=batch.lengths[sl].contiguous(), accept_u=batch.accept_u[sl].contiguous(),
                sample_u=batch.sample_u[sl].contiguous(),
                draft_u=torch.rand((steps, self.L, n, 1), generator=g, device=dev),
                tok=torch.empty((self.L, n, 1), dtype=torch.int32, device=dev),
                status=torch.zeros(1, dtype=torch.int32, device=dev),
                out=binding.Outputs("multidraft", self.B, self.K, self.L, self.V, dev)))
        self.s_draft = torch.cuda.Stream(device=dev)
        self.s_verify = torch.cuda.Stream(device=dev)

    # ---------------------------------------------------------------- phases
    def draft(self, h: int, step: int, stream) -> None:
        """The draft phase of half h: a token per draft and depth."""
        x = self.halves[h]
        n = self.B * self.K
        for j in range(self.L):
            rows = x.draft[:, :, j, :].reshape(n, x.draft.shape[-1])
            binding.sample_rows(rows, 1, x.draft_u[step % self.steps, j], self.T, V=self.V, tokens=x.tok[j],
                                device_status=x.status, stream=stream)
        with torch.cuda.stream(stream):
            x.tokens.copy_(x.tok.view(self.L, self.B, self.K).permute(1, 2, 0))

    def verify(self, h: int, stream) -> None:
        """The verify phase of half h."""
        x = self.halves[h]
        binding.verify("multidraft", x.target, x.draft, x.tokens, x.lengths, x.accept_u, x.sample_u, self.T,
                       V=self.V, out=x.out, stream=stream)

    # ----------------------------------------------------------------- steps
    def step_overlapped(self, step: int) -> None:
        """Half v verifies on one stream while half d drafts on the other;
        the caller's stream waits for both."""
        v, d = roles(step)
        cur = torch.cuda.current_stream()
        start = torch.cuda.Event()
        start.record(cur)
        self.s_verify.wait_event(start)
        self.s_draft.wait_event(start)
        self.verify(v, self.s_verify)
        self.draft(d, step, self.s_draft)
        cur.wait_stream(self.s_verify)
        cur.wait_stream(self.s_draft)

    def step_sequential(self, step: int) -> None:
        """The same work on the caller's stream: draft, then verify."""
        v, d = roles(step)
        cur = torch.cuda.current_stream()
        self.draft(d, step, cur)
        self.verify(v, cur)

    def results(self, h: int):
        """Host copies of half h's last verification outputs and draft tokens."""
        x = self.halves[h]
        return {"accept_len": x.out.accept_len.cpu(), "accept_draft": x.out.accept_draft.cpu(),
                "out_token": x.out.out_token.cpu(), "tokens": x.tokens.cpu(),
                "device_status": int(x.out.device_status.item()) | int(x.status.item())}


def time_ms(fn, reps: int, stream: Optional[torch.cuda.Stream] = None) -> float:
    """Median milliseconds of fn() over reps calls, CUDA events on the
    caller's stream (fn joins any side streams into it)."""
    stream = stream or torch.cuda.current_stream()
    ts = []
    for i in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn(i)
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    ts.sort()
    return ts[len(ts) // 2]


def measure(emu: PsdEmulator, reps: int = 10, warmup: int = 3):
    """Phase and step times (ms, medians) and the share of the shorter phase
    the overlap hides."""
    for i in range(warmup):
        emu.step_overlapped(i)
        emu.step_sequential(i)
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    t_draft = time_ms(lambda i: emu.draft(1, i, cur), reps)
    t_verify = time_ms(lambda i: emu.verify(0, cur), reps)
    t_seq = time_ms(emu.step_sequential, reps)
    t_psd = time_ms(emu.step_overlapped, reps)
    return {"draft_ms": t_draft, "verify_ms": t_verify, "sequential_step_ms": t_seq, "psd_step_ms": t_psd,
            "hidden_fraction": hidden_fraction(t_draft, t_verify, t_seq, t_psd),
            "step_time_saved": 1.0 - t_psd / t_seq if t_seq > 0 else 0.0}
