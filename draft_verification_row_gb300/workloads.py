"""Seeded synthetic verification batches.

The pages measure on model outputs over public datasets, none of which are
available here; these batches stand in for them with the shapes the pages'
workloads have (vocabularies of 32000, 128256 and 151936 tokens, batches up
to 256 requests, up to 8 drafts of up to 8 tokens) and logit statistics
chosen to spread acceptance rates.

This module only produces inputs.  It holds none of the verification
arithmetic: the drafted tokens are drawn from the draft softmax the way a
draft model would draw them, with torch's own sampler.  Both the CUDA path
and the CPU oracle take their inputs from here.

Layout (the library's): target [B][K][L+1][stride], draft [B][K][L][stride],
tokens [B][K][L] int32, lengths [B] int32, accept_u [B][K][L] and
sample_u [B][K][L+1] fp32 uniforms in [0, 1).  Row (b, k, j) holds the
logits conditioned on draft k's first j tokens, so drafts sharing a prefix
get identical rows (row 0, the context, is shared by every draft).
Columns past V in a row (stride padding) hold NaN: they are never read.
"""
from dataclasses import dataclass, field
from typing import Optional

import torch

# Named workloads.  noise is the std of the draft's deviation from the
# target logits (a (lo, hi) pair draws one std per request, uniformly).
WORKLOADS = {
    "token-B4-K1-L4-V1024-f32": dict(
        B=4, K=1, L=4, V=1024, dtype="f32", T=1.0, temps=(1.0,),
        target_std=2.0, noise=0.5, spikes=0, spike_height=0.0, zipf=0.0, ragged=False, seed=1001),
    "token-greedy-B64-K1-L5-V32000-bf16": dict(
        B=64, K=1, L=5, V=32000, dtype="bf16", T=1.0, temps=(0.0, 1.0),
        target_std=3.0, noise=1.0, spikes=20, spike_height=8.0, zipf=0.0, ragged=False, seed=1002),
    "block-B128-K1-L5-V128256-bf16": dict(
        B=128, K=1, L=5, V=128256, dtype="bf16", T=0.7, temps=(0.7,),
        target_std=3.0, noise=(0.3, 2.0), spikes=0, spike_height=0.0, zipf=0.0, ragged=False, seed=1003),
    "multidraft-B32-K4-L4-V32000-f32": dict(
        B=32, K=4, L=4, V=32000, dtype="f32", T=0.7, temps=(0.1, 0.4, 0.7),
        target_std=2.0, noise=0.8, spikes=0, spike_height=0.0, zipf=0.0, ragged=False, seed=1004),
    "mixed-B256-K8-L8-V151936-bf16": dict(
        B=256, K=8, L=8, V=151936, dtype="bf16", T=0.7, temps=(0.7,),
        target_std=3.0, noise=1.0, spikes=0, spike_height=0.0, zipf=1.1, ragged=True, seed=1005),
}

# the large mixed batch is the throughput workload
HEADLINE = "mixed-B256-K8-L8-V151936-bf16"


@dataclass
class Batch:
    name: str
    B: int
    K: int
    L: int
    V: int
    stride: int
    dtype: str                 # "f32" or "bf16"
    temperature: float
    target: torch.Tensor
    draft: torch.Tensor
    tokens: torch.Tensor
    lengths: torch.Tensor
    accept_u: torch.Tensor
    sample_u: torch.Tensor
    meta: dict = field(default_factory=dict)

    def to(self, device):
        kw = {k: getattr(self, k) for k in ("name", "B", "K", "L", "V", "stride", "dtype", "temperature")}
        for k in ("target", "draft", "tokens", "lengths", "accept_u", "sample_u"):
            kw[k] = getattr(self, k).to(device)
        return Batch(meta=dict(self.meta), **kw)

    @property
    def positions(self) -> int:
        """Verified draft positions: sum over requests of K * L_b."""
        return int(self.lengths.to(torch.int64).sum().item()) * self.K


def _round8(n):
    return (n + 7) // 8 * 8


def make(workload, device="cpu", *, seed: Optional[int] = None, temperature: Optional[float] = None,
         B: Optional[int] = None, K: Optional[int] = None, L: Optional[int] = None,
         V: Optional[int] = None, dtype: Optional[str] = None, stride_pad: int = 0,
         lengths=None, poison_unread: bool = False) -> Batch:
    """Generate one batch of a named workload (or a dict of the same keys).

    Keyword overrides change the shape for small parity cases.  With
    ``poison_unread`` every row the method never reads (rows past a
    request's length, duplicate copies of a shared prefix's rows) is filled
    with NaN and padding tokens with -1, so that reading any of them shows.
    """
    cfg = dict(WORKLOADS[workload]) if isinstance(workload, str) else dict(workload)
    name = workload if isinstance(workload, str) else cfg.get("name", "custom")
    for k, v in (("B", B), ("K", K), ("L", L), ("V", V), ("dtype", dtype)):
        if v is not None:
            cfg[k] = v
    B_, K_, L_, V_ = cfg["B"], cfg["K"], cfg["L"], cfg["V"]
    # the C interface takes the temperature as a float: the batch carries
    # that float's value, so that every consumer is handed the same number
    T = float(torch.tensor(cfg["T"] if temperature is None else float(temperature), dtype=torch.float32))
    seed = cfg["seed"] if seed is None else seed
    dt = torch.bfloat16 if cfg["dtype"] == "bf16" else torch.float32
    stride = _round8(V_) + stride_pad
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))

    tgt = torch.full((B_, K_, L_ + 1, stride), float("nan"), dtype=dt, device=dev)
    dft = torch.full((B_, K_, L_, stride), float("nan"), dtype=dt, device=dev)
    tokens = torch.zeros((B_, K_, L_), dtype=torch.int32, device=dev)
    if lengths is not None:
        lens = torch.as_tensor(lengths, dtype=torch.int32, device=dev).clone()
    elif cfg["ragged"] and L_ > 0:
        lens = torch.randint(1, L_ + 1, (B_,), generator=g, device=dev, dtype=torch.int64).to(torch.int32)
    else:
        lens = torch.full((B_,), L_, dtype=torch.int32, device=dev)
    noise = cfg["noise"]
    if isinstance(noise, (tuple, list)):
        lo, hi = noise
        nstd = lo + (hi - lo) * torch.rand(B_, generator=g, device=dev)
    else:
        nstd = torch.full((B_,), float(noise), device=dev)

    owners = []
    for j in range(L_ + 1):
        t = torch.randn(B_, K_, V_, generator=g, device=dev) * cfg["target_std"]
        if cfg["spikes"]:
            idx = torch.rand(B_ * K_, V_, generator=g, device=dev).topk(cfg["spikes"], dim=1).indices
            t.view(B_ * K_, V_).scatter_add_(
                1, idx, torch.full(idx.shape, float(cfg["spike_height"]), device=dev))
        if cfg["zipf"]:
            rank = torch.rand(B_ * K_, V_, generator=g, device=dev).argsort(dim=1)
            t += (-cfg["zipf"] * torch.log(rank.to(torch.float32) + 1.0)).view(B_, K_, V_)
        d = t + torch.randn(B_, K_, V_, generator=g, device=dev) * nstd[:, None, None]
        # drafts that share their first j tokens share the node's rows
        if j == 0:
            owner = torch.zeros((B_, K_), dtype=torch.int64, device=dev)
        else:
            pre = tokens[:, :, :j]
            same = (pre[:, :, None, :] == pre[:, None, :, :]).all(dim=-1)   # [B, k, k']
            owner = same.to(torch.int8).argmax(dim=-1)                         # first k' sharing k's prefix
        owners.append(owner)
        gidx = owner[:, :, None].expand(B_, K_, V_)
        tq = t.gather(1, gidx).to(dt)
        dq = d.gather(1, gidx).to(dt)
        tgt[:, :, j, :V_] = tq
        if j < L_:
            dft[:, :, j, :V_] = dq
            if T > 0:
                probs = torch.softmax(dq.to(torch.float32) / T, dim=-1).view(B_ * K_, V_)
                x = torch.multinomial(probs, 1, generator=g).view(B_, K_)
            else:
                x = dq.to(torch.float32).argmax(dim=-1)
            tokens[:, :, j] = x.to(torch.int32)
    accept_u = torch.rand((B_, K_, L_), generator=g, device=dev)
    sample_u = torch.rand((B_, K_, L_ + 1), generator=g, device=dev)

    if poison_unread:
        nan = float("nan")
        ar = torch.arange(L_ + 1, device=dev)
        past_t = ar[None, :] > lens[:, None].to(torch.int64)            # [B, L+1]
        tgt[past_t[:, None, :, None].expand_as(tgt)] = nan
        if L_ > 0:
            past_d = ar[None, :L_] >= lens[:, None].to(torch.int64)     # [B, L]
            dft[past_d[:, None, :, None].expand_as(dft)] = nan
            tokens[past_d[:, None, :].expand_as(tokens)] = -1
        for j, owner in enumerate(owners):
            dup = owner != torch.arange(K_, device=dev)[None, :]           # [B, K]
            tgt[:, :, j][dup] = nan
            if j < L_:
                dft[:, :, j][dup] = nan

    meta = {k: cfg[k] for k in ("target_std", "noise", "spikes", "spike_height", "zipf", "ragged")}
    meta["seed"] = int(seed)
    return Batch(name=name, B=B_, K=K_, L=L_, V=V_, stride=stride, dtype=cfg["dtype"], temperature=T,
                 target=tgt, draft=dft, tokens=tokens, lengths=lens, accept_u=accept_u,
                 sample_u=sample_u, meta=meta)


# ---------------------------------------------------------------------------
# Greedy verification fused into the target model's LM head: the inputs are
# the target model's final hidden states and its LM head instead of logits.

LM_HEAD_WORKLOADS = {
    # the mixed batch's shape with a hidden size of 4096 (8B-class models
    # with this vocabulary size)
    "lmhead-greedy-B256-K8-L8-V151936-d4096": dict(
        B=256, K=8, L=8, V=151936, d=4096, logit_std=3.0, agree=0.6, ragged=True, seed=1006),
}

LM_HEAD_HEADLINE = "lmhead-greedy-B256-K8-L8-V151936-d4096"


@dataclass
class LmHeadBatch:
    name: str
    B: int
    K: int
    L: int
    V: int
    d: int
    hidden: torch.Tensor   # [B][K][L+1][d] bf16
    lm_head: torch.Tensor  # [V][d] bf16
    tokens: torch.Tensor   # [B][K][L] int32
    lengths: torch.Tensor  # [B] int32
    meta: dict = field(default_factory=dict)

    def to(self, device):
        kw = {k: getattr(self, k) for k in ("name", "B", "K", "L", "V", "d")}
        for k in ("hidden", "lm_head", "tokens", "lengths"):
            kw[k] = getattr(self, k).to(device)
        return LmHeadBatch(meta=dict(self.meta), **kw)

    @property
    def positions(self) -> int:
        return int(self.lengths.to(torch.int64).sum().item()) * self.K


def make_lm_head(workload, device="cpu", *, seed: Optional[int] = None, B: Optional[int] = None,
                 K: Optional[int] = None, L: Optional[int] = None, V: Optional[int] = None,
                 d: Optional[int] = None, lengths=None, integer: int = 0, poison_unread: bool = False,
                 agree: Optional[float] = None) -> LmHeadBatch:
    """One batch for greedy verification fused into the LM head.

    W ~ N(0, logit_std^2 / d) and hidden ~ N(0, 1), so logits have std about
    logit_std.  Drafts are built depth by depth like a greedy draft model
    that agrees with the target: draft k's next token is the target row's
    argmax (found with torch) with probability ``agree``, else a uniform
    token; drafts sharing a prefix share its hidden row.  ``integer`` > 0
    draws every entry of hidden and W uniformly from -integer..integer
    instead (exact logits, many ties).  With ``poison_unread`` the rows the
    method never reads (past a request's length, duplicate copies of a
    shared prefix's row) hold NaN.
    """
    cfg = dict(LM_HEAD_WORKLOADS[workload]) if isinstance(workload, str) else dict(workload)
    name = workload if isinstance(workload, str) else cfg.get("name", "custom")
    for k, v in (("B", B), ("K", K), ("L", L), ("V", V), ("d", d), ("agree", agree)):
        if v is not None:
            cfg[k] = v
    B_, K_, L_, V_, d_ = cfg["B"], cfg["K"], cfg["L"], cfg["V"], cfg["d"]
    seed = cfg["seed"] if seed is None else seed
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))

    def draw(*shape, scale=1.0):
        if integer:
            return torch.randint(-integer, integer + 1, shape, generator=g, device=dev).to(torch.float32)
        return torch.randn(*shape, generator=g, device=dev) * scale

    W = draw(V_, d_, scale=cfg["logit_std"] / d_ ** 0.5).to(torch.bfloat16)
    Wf = W.to(torch.float32)
    hidden = torch.empty((B_, K_, L_ + 1, d_), dtype=torch.bfloat16, device=dev)
    tokens = torch.zeros((B_, K_, L_), dtype=torch.int32, device=dev)
    if lengths is not None:
        lens = torch.as_tensor(lengths, dtype=torch.int32, device=dev).clone()
    elif cfg["ragged"] and L_ > 0:
        lens = torch.randint(1, L_ + 1, (B_,), generator=g, device=dev, dtype=torch.int64).to(torch.int32)
    else:
        lens = torch.full((B_,), L_, dtype=torch.int32, device=dev)
    owners = []
    for j in range(L_ + 1):
        h = draw(B_, K_, d_).to(torch.bfloat16)
        if j == 0:
            owner = torch.zeros((B_, K_), dtype=torch.int64, device=dev)
        else:
            pre = tokens[:, :, :j]
            same = (pre[:, :, None, :] == pre[:, None, :, :]).all(dim=-1)
            owner = same.to(torch.int8).argmax(dim=-1)
        owners.append(owner)
        h = h.gather(1, owner[:, :, None].expand(B_, K_, d_))
        hidden[:, :, j] = h
        if j < L_:
            rows = h.reshape(B_ * K_, d_).to(torch.float32)
            am = torch.zeros(0, dtype=torch.int64, device=dev)
            if B_ * K_:
                am = torch.cat([(rows[i:i + 512] @ Wf.T).argmax(dim=-1) for i in range(0, B_ * K_, 512)])
            pick = torch.rand(B_ * K_, generator=g, device=dev) < cfg["agree"]
            other = torch.randint(0, V_, (B_ * K_,), generator=g, device=dev)
            tokens[:, :, j] = torch.where(pick, am, other).view(B_, K_).to(torch.int32)

    if poison_unread:
        nan = float("nan")
        ar = torch.arange(L_ + 1, device=dev)
        past = ar[None, :] > lens[:, None].to(torch.int64)
        hidden[past[:, None, :, None].expand_as(hidden)] = nan
        if L_ > 0:
            past_d = ar[None, :L_] >= lens[:, None].to(torch.int64)
            tokens[past_d[:, None, :].expand_as(tokens)] = -1
        for j, owner in enumerate(owners):
            dup = owner != torch.arange(K_, device=dev)[None, :]
            hidden[:, :, j][dup] = nan

    meta = {k: cfg[k] for k in ("logit_std", "agree", "ragged")}
    meta.update(seed=int(seed), integer=int(integer))
    return LmHeadBatch(name=name, B=B_, K=K_, L=L_, V=V_, d=d_, hidden=hidden, lm_head=W, tokens=tokens,
                       lengths=lens, meta=meta)
