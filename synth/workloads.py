"""The five synthetic workloads of the verify step, drawn from a seeded torch
generator on any device.

Shapes and value distributions follow the serving workloads the pages
describe (Llama-3 / Qwen sized vocabularies, N = 3..7 draft tokens); no
dataset, model or prompt is involved.  Everything is reproducible from
(config, seed, device).

Recipe (per sequence b, position i, token k):
  base[b,i,k] ~ N(0, sigma_p^2) for i = 0..N       (draft-side logits)
  draft[b,i,:] = base[b,i,:]                        for i = 0..N-1
  target[b,i,:] = base[b,i,:] + N(0, sigma_q^2)     for i = 0..N
then the per-config twists below, then rounding to the storage dtype.
Draft tokens are drawn from the draft's own distribution at temperature T by
the Gumbel-max trick on the stored logits (argmax of z/T + Gumbel noise),
which draws exactly from softmax(z/T) without evaluating it; for T <= 0 the
draft is the argmax.  Uniforms are U[0,1) float32, one per accept test
(columns 0..N-1) and one for the final residual/bonus sample (column N).
"""
from __future__ import annotations

import dataclasses

import torch

# name -> parameters.  "tiny" and "small" are latency cases, "mixed" runs the
# greedy and sampled paths side by side, "headline" is the Qwen-vocabulary
# batch that the roofline is reported on, "stress" is the float32 batch with
# forced near-zero-probability drafts.
CONFIGS = {
    "tiny": dict(B=1, N=4, V=1024, dtype="f32", T=1.0, sigma_p=2.0, sigma_q=1.0),
    "small": dict(B=8, N=5, V=32000, dtype="bf16", T=1.0, sigma_p=3.0, sigma_q=0.5,
                  spike_frac=0.10, spike=8.0),
    "mixed": dict(B=64, N=5, V=128256, dtype="bf16", T=(0.0, 0.7, 1.0), sigma_p=3.0,
                  sigma_q=(0.3, 2.0)),
    "headline": dict(B=256, N=7, V=151936, dtype="bf16", T=0.8, sigma_p=3.0, sigma_q=1.0,
                     zipf=1.1),
    "stress": dict(B=1024, N=3, V=128256, dtype="f32", T=1.0, sigma_p=2.0, sigma_q=1.5,
                   force_frac=0.05, force_logit=-30.0),
}


def config(name: str, **overrides) -> dict:
    c = dict(CONFIGS[name])
    c.update(overrides)
    c["name"] = name
    return c


@dataclasses.dataclass
class Workload:
    name: str
    B: int
    N: int
    V: int
    dtype: str               # "bf16" or "f32"
    target: torch.Tensor     # [B, N+1, V]
    draft: torch.Tensor      # [B, N, V]
    draft_tokens: torch.Tensor  # [B, N] int32
    uniforms: torch.Tensor   # [B, N+1] float32
    temperature: torch.Tensor  # [B] float32
    greedy: bool = False

    @property
    def elt(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    @property
    def verified_rows(self) -> int:
        return self.B * (self.N + 1)

    @property
    def logit_bytes(self) -> int:
        return self.B * (2 * self.N + 1) * self.V * self.elt

    def to(self, device) -> "Workload":
        d = dataclasses.replace(self)
        for f in ("target", "draft", "draft_tokens", "uniforms", "temperature"):
            setattr(d, f, getattr(self, f).to(device))
        return d


def _torch_dtype(name: str):
    return torch.bfloat16 if name == "bf16" else torch.float32


def make_workload(name: str, seed: int = 0, device="cpu", chunk_rows: int = 4096,
                  **overrides) -> Workload:
    """Draw one workload.  ``overrides`` may change B, N, V, dtype, T ... of
    the named config (used for reduced-size parity cases)."""
    c = config(name, **overrides)
    B, N, V = c["B"], c["N"], c["V"]
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    tdt = _torch_dtype(c["dtype"])

    # per-sequence temperature and target noise scale
    T_spec = c["T"]
    if isinstance(T_spec, tuple):
        pick = torch.randint(0, len(T_spec), (B,), generator=g, device=dev)
        T = torch.tensor(T_spec, dtype=torch.float32, device=dev)[pick]
    else:
        T = torch.full((B,), float(T_spec), dtype=torch.float32, device=dev)
    sq_spec = c["sigma_q"]
    if isinstance(sq_spec, tuple):
        lo, hi = sq_spec
        sigma_q = lo + (hi - lo) * torch.rand((B,), generator=g, device=dev)
    else:
        sigma_q = torch.full((B,), float(sq_spec), device=dev)

    target = torch.empty((B, N + 1, V), dtype=tdt, device=dev)
    draft = torch.empty((B, N, V), dtype=tdt, device=dev)

    zipf_bias = None
    if c.get("zipf"):
        rank = torch.arange(1, V + 1, device=dev, dtype=torch.float32)
        zipf_bias = -float(c["zipf"]) * torch.log(rank)

    # generate a few sequences at a time to bound temporaries
    per = max(1, chunk_rows // (N + 1))
    for b0 in range(0, B, per):
        b1 = min(B, b0 + per)
        nb = b1 - b0
        base = torch.randn((nb, N + 1, V), generator=g, device=dev) * c["sigma_p"]
        noise = torch.randn((nb, N + 1, V), generator=g, device=dev)
        zq = base + noise * sigma_q[b0:b1].view(nb, 1, 1)
        if zipf_bias is not None:
            odd = (torch.arange(b0, b1, device=dev) % 2 == 1).view(nb, 1, 1)
            base = torch.where(odd, base + zipf_bias, base)
            zq = torch.where(odd, zq + zipf_bias, zq)
        target[b0:b1] = zq.to(tdt)
        draft[b0:b1] = base[:, :N].to(tdt)
        del base, noise, zq

    # spiky target rows: one uniformly chosen token gets +spike
    if c.get("spike_frac"):
        rows = torch.rand((B, N + 1), generator=g, device=dev) < c["spike_frac"]
        tok = torch.randint(0, V, (B, N + 1), generator=g, device=dev)
        idx = rows.nonzero(as_tuple=False)
        if idx.numel():
            bb, ii = idx[:, 0], idx[:, 1]
            kk = tok[bb, ii]
            vals = target[bb, ii, kk].float() + float(c["spike"])
            target[bb, ii, kk] = vals.to(tdt)

    # draft tokens: Gumbel-max on the stored draft logits at temperature T
    tokens = torch.empty((B, N), dtype=torch.int32, device=dev)
    for b0 in range(0, B, per):
        b1 = min(B, b0 + per)
        z = draft[b0:b1].float()
        Tb = T[b0:b1].view(-1, 1, 1)
        gumbel = -torch.log(torch.empty_like(z).exponential_(generator=g))
        sampled = torch.argmax(z / torch.where(Tb > 0, Tb, torch.ones_like(Tb)) + gumbel, dim=-1)
        greedy = torch.argmax(z, dim=-1)
        tokens[b0:b1] = torch.where(Tb.view(-1, 1) > 0, sampled, greedy).to(torch.int32)
        del z, gumbel

    # forced drafts on tokens the target gives (almost) no mass
    if c.get("force_frac") and N > 0:
        hit = torch.rand((B, N), generator=g, device=dev) < c["force_frac"]
        tok = torch.randint(0, V, (B, N), generator=g, device=dev)
        idx = hit.nonzero(as_tuple=False)
        if idx.numel():
            bb, ii = idx[:, 0], idx[:, 1]
            kk = tok[bb, ii]
            target[bb, ii, kk] = torch.tensor(float(c["force_logit"]), dtype=tdt, device=dev)
            tokens[bb, ii] = kk.to(torch.int32)

    uniforms = torch.rand((B, N + 1), generator=g, device=dev, dtype=torch.float32)
    return Workload(name=name, B=B, N=N, V=V, dtype=c["dtype"], target=target, draft=draft,
                    draft_tokens=tokens, uniforms=uniforms, temperature=T)


# ---- candidate trees ---------------------------------------------------------
#
# Tree recipe (per sequence b, node n = 0..M, node 0 = the committed context):
#   base[b,n,:] ~ N(0, sigma_p^2)              (the draft's logits at node n)
#   draft[b,n,:] = base[b,n,:];  target[b,n,:] = base[b,n,:] + N(0, sigma_q^2)
# then the twists, then rounding to the storage dtype.  The children of node n
# are independent Gumbel-max draws from softmax(draft[b,n,:]/T) (argmax for
# T <= 0).  Topologies: "eagle16" is a fixed 16-node tree shaped like the
# static trees of Medusa / EAGLE (wide at the root, narrowing with depth);
# "random" gives every sequence its own tree, parent[n] uniform in
# [max(0, n-3), n-1] (dynamic trees, as in EAGLE-2).  Uniforms: one per node
# (column n >= 1: the accept test of node n; column 0: the final sample).
EAGLE16_PARENT = [-1, 0, 0, 0, 0, 1, 1, 1, 2, 2, 3, 5, 5, 6, 8, 11]

TREE_CONFIGS = {
    "tree_small": dict(B=6, M=10, V=4096, dtype="f32", T=1.0, sigma_p=2.0, sigma_q=1.0, topology="random"),
    "tree_mixed": dict(B=16, M=20, V=32000, dtype="bf16", T=(0.0, 0.7, 1.0), sigma_p=3.0, sigma_q=(0.3, 2.0),
                       topology="random", spike_frac=0.10, spike=8.0),
    "tree": dict(B=64, M=15, V=151936, dtype="bf16", T=0.8, sigma_p=3.0, sigma_q=1.0, zipf=1.1,
                 topology="eagle16"),
}


@dataclasses.dataclass
class TreeWorkload:
    name: str
    B: int
    M: int
    V: int
    dtype: str
    target: torch.Tensor       # [B, M+1, V]
    draft: torch.Tensor        # [B, M+1, V] (rows of leaves are not read)
    parent: torch.Tensor       # [B, M+1] int32
    tokens: torch.Tensor       # [B, M+1] int32 (column 0 unused)
    uniforms: torch.Tensor     # [B, M+1] float32
    temperature: torch.Tensor  # [B] float32
    greedy: bool = False

    @property
    def elt(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def internal(self):
        """[B, M+1] bool: nodes with at least one child."""
        has = torch.zeros((self.B, self.M + 1), dtype=torch.bool, device=self.parent.device)
        if self.M > 0:
            has.scatter_(1, self.parent[:, 1:].long().clamp(min=0), True)
        return has

    @property
    def logit_bytes(self) -> int:
        """Rows the verify reads: every target row, the draft rows of internal
        nodes (of sampled sequences)."""
        sampled = self.temperature > 0 if not self.greedy else torch.zeros_like(self.temperature, dtype=torch.bool)
        draft_rows = int((self.internal() & sampled.view(-1, 1)).sum())
        return (self.B * (self.M + 1) + draft_rows) * self.V * self.elt


def tree_config(name: str, **overrides) -> dict:
    c = dict(TREE_CONFIGS[name])
    c.update(overrides)
    c["name"] = name
    return c


def make_tree_workload(name: str, seed: int = 0, device="cpu", **overrides) -> TreeWorkload:
    c = tree_config(name, **overrides)
    B, M, V = c["B"], c["M"], c["V"]
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed) + 7919)
    tdt = _torch_dtype(c["dtype"])

    T_spec = c["T"]
    if isinstance(T_spec, tuple):
        pick = torch.randint(0, len(T_spec), (B,), generator=g, device=dev)
        T = torch.tensor(T_spec, dtype=torch.float32, device=dev)[pick]
    else:
        T = torch.full((B,), float(T_spec), dtype=torch.float32, device=dev)
    sq_spec = c["sigma_q"]
    if isinstance(sq_spec, tuple):
        lo, hi = sq_spec
        sigma_q = lo + (hi - lo) * torch.rand((B,), generator=g, device=dev)
    else:
        sigma_q = torch.full((B,), float(sq_spec), device=dev)

    if c["topology"] == "eagle16":
        assert M == len(EAGLE16_PARENT) - 1
        parent = torch.tensor(EAGLE16_PARENT, dtype=torch.int32, device=dev).repeat(B, 1)
    else:
        parent = torch.full((B, M + 1), -1, dtype=torch.int32, device=dev)
        for n in range(1, M + 1):
            lo = max(0, n - 3)
            parent[:, n] = torch.randint(lo, n, (B,), generator=g, device=dev).to(torch.int32)

    target = torch.empty((B, M + 1, V), dtype=tdt, device=dev)
    draft = torch.empty((B, M + 1, V), dtype=tdt, device=dev)
    zipf_bias = None
    if c.get("zipf"):
        rank = torch.arange(1, V + 1, device=dev, dtype=torch.float32)
        zipf_bias = -float(c["zipf"]) * torch.log(rank)
    per = max(1, 4096 // (M + 1))
    for b0 in range(0, B, per):
        b1 = min(B, b0 + per)
        nb = b1 - b0
        base = torch.randn((nb, M + 1, V), generator=g, device=dev) * c["sigma_p"]
        zq = base + torch.randn((nb, M + 1, V), generator=g, device=dev) * sigma_q[b0:b1].view(nb, 1, 1)
        if zipf_bias is not None:
            odd = (torch.arange(b0, b1, device=dev) % 2 == 1).view(nb, 1, 1)
            base = torch.where(odd, base + zipf_bias, base)
            zq = torch.where(odd, zq + zipf_bias, zq)
        target[b0:b1] = zq.to(tdt)
        draft[b0:b1] = base.to(tdt)
        del base, zq

    if c.get("spike_frac"):
        rows = torch.rand((B, M + 1), generator=g, device=dev) < c["spike_frac"]
        tok = torch.randint(0, V, (B, M + 1), generator=g, device=dev)
        idx = rows.nonzero(as_tuple=False)
        if idx.numel():
            bb, nn = idx[:, 0], idx[:, 1]
            kk = tok[bb, nn]
            target[bb, nn, kk] = (target[bb, nn, kk].float() + float(c["spike"])).to(tdt)

    # children: independent Gumbel-max draws from their parent's draft row
    tokens = torch.zeros((B, M + 1), dtype=torch.int32, device=dev)
    for n in range(1, M + 1):
        par = parent[:, n].long()
        z = draft[torch.arange(B, device=dev), par].float()
        Tb = T.view(-1, 1)
        gumbel = -torch.log(torch.empty_like(z).exponential_(generator=g))
        sampled = torch.argmax(z / torch.where(Tb > 0, Tb, torch.ones_like(Tb)) + gumbel, dim=-1)
        greedy = torch.argmax(z, dim=-1)
        tokens[:, n] = torch.where(T > 0, sampled, greedy).to(torch.int32)
    uniforms = torch.rand((B, M + 1), generator=g, device=dev, dtype=torch.float32)
    return TreeWorkload(name=name, B=B, M=M, V=V, dtype=c["dtype"], target=target, draft=draft, parent=parent,
                        tokens=tokens, uniforms=uniforms, temperature=T)


# ---- hidden states and LM heads (the fused path) ---------------------------------
#
# Recipe: verifier weight W_t [V, Kt] ~ N(0, (sigma_z^2 / Kt)), hidden states
# h_t [B*(N+1), Kt] ~ N(0, 1), so the verifier logits h_t W_t^T have standard
# deviation ~ sigma_z.  The draft model reads the first Kd features:
# W_d = W_t[:, :Kd] * sqrt(Kt / Kd) and h_d[b*N+i] = h_t[b*(N+1)+i, :Kd] +
# N(0, rho^2), so draft and verifier logits correlate (about sqrt(Kd/Kt)).
# Draft tokens: Gumbel-max draws from the draft's own logits at temperature T
# (argmax at T <= 0); uniforms U[0, 1).  All tensors bf16 except the uniforms.
FUSED_CONFIGS = {
    "fused_small": dict(B=8, N=3, V=4096, Kt=256, Kd=128, T=1.0, sigma_z=3.0, rho=0.3),
    "fused_mixed": dict(B=16, N=4, V=32000, Kt=512, Kd=256, T=(0.0, 0.7, 1.0), sigma_z=3.0, rho=0.5),
    "fused": dict(B=256, N=7, V=151936, Kt=3584, Kd=896, T=0.8, sigma_z=3.0, rho=0.3),
}


@dataclasses.dataclass
class FusedWorkload:
    name: str
    B: int
    N: int
    V: int
    Kt: int
    Kd: int
    target_hidden: torch.Tensor   # [B*(N+1), Kt] bf16
    target_weight: torch.Tensor   # [V, Kt] bf16
    draft_hidden: torch.Tensor    # [B*N, Kd] bf16
    draft_weight: torch.Tensor    # [V, Kd] bf16
    draft_tokens: torch.Tensor    # [B, N] int32
    uniforms: torch.Tensor        # [B, N+1] float32
    temperature: torch.Tensor     # [B] float32
    greedy: bool = False

    @property
    def flops(self) -> int:
        return 2 * self.V * (self.B * (self.N + 1) * self.Kt + self.B * self.N * self.Kd)


def make_fused_workload(name: str, seed: int = 0, device="cpu", **overrides) -> FusedWorkload:
    c = dict(FUSED_CONFIGS[name])
    c.update(overrides)
    B, N, V, Kt, Kd = c["B"], c["N"], c["V"], c["Kt"], c["Kd"]
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed) + 104729)
    T_spec = c["T"]
    if isinstance(T_spec, tuple):
        pick = torch.randint(0, len(T_spec), (B,), generator=g, device=dev)
        T = torch.tensor(T_spec, dtype=torch.float32, device=dev)[pick]
    else:
        T = torch.full((B,), float(T_spec), dtype=torch.float32, device=dev)
    wt = torch.empty((V, Kt), dtype=torch.bfloat16, device=dev)
    step = 8192
    for v0 in range(0, V, step):
        v1 = min(V, v0 + step)
        wt[v0:v1] = (torch.randn((v1 - v0, Kt), generator=g, device=dev) * (c["sigma_z"] / Kt ** 0.5)).to(torch.bfloat16)
    wd = (wt[:, :Kd].float() * (Kt / Kd) ** 0.5).to(torch.bfloat16).contiguous()
    ht = torch.randn((B, N + 1, Kt), generator=g, device=dev)
    hd = ht[:, :N, :Kd] + torch.randn((B, N, Kd), generator=g, device=dev) * c["rho"]
    ht = ht.reshape(B * (N + 1), Kt).to(torch.bfloat16).contiguous()
    hd = hd.reshape(B * N, Kd).to(torch.bfloat16).contiguous()
    tokens = torch.empty((B, N), dtype=torch.int32, device=dev)
    for b0 in range(0, B, 32):
        b1 = min(B, b0 + 32)
        zd = (hd[b0 * N:b1 * N].float() @ wd.float().T).view(b1 - b0, N, V)  # the draft's logits, to draw its tokens
        Tb = T[b0:b1].view(-1, 1, 1)
        gumbel = -torch.log(torch.empty_like(zd).exponential_(generator=g))
        sampled = torch.argmax(zd / torch.where(Tb > 0, Tb, torch.ones_like(Tb)) + gumbel, dim=-1)
        tokens[b0:b1] = torch.where(Tb.view(-1, 1) > 0, sampled, torch.argmax(zd, dim=-1)).to(torch.int32)
        del zd, gumbel
    uniforms = torch.rand((B, N + 1), generator=g, device=dev, dtype=torch.float32)
    return FusedWorkload(name, B, N, V, Kt, Kd, ht, wt, hd, wd, tokens, uniforms, T)


def describe(name: str) -> str:
    c = config(name)
    B, N, V = c["B"], c["N"], c["V"]
    elt = 2 if c["dtype"] == "bf16" else 4
    gb = B * (2 * N + 1) * V * elt / 1e9
    return f"{name}: B={B} N={N} V={V} {c['dtype']} ({gb:.3f} GB of logits)"


__all__ = ["CONFIGS", "Workload", "config", "make_workload", "describe", "TREE_CONFIGS", "TreeWorkload",
           "tree_config", "make_tree_workload", "EAGLE16_PARENT", "FUSED_CONFIGS", "FusedWorkload",
           "make_fused_workload"]
