"""Seeded generator of verification inputs (CPU, torch).

Recipe per sequence b of step s (each sequence has its own seeds, so any subset
of a batch can be regenerated on its own):

* target logits: fp32 normals N(0, target_std^2) for the K+1 target rows; when
  the workload asks for peaks, `peaks` distinct random ids per target row get
  `+peak_boost`;
* draft logits: draft row t = target row t (peaks included) + N(0, noise^2),
  t < K (the draft row conditions on the same prefix as target row t);
* both are then rounded to the workload dtype (bf16 rounds to nearest even);
* draft tokens: x_t = argmax_i(dl[t,i]/T + G_i), G_i standard Gumbel noise in
  fp64 drawn from a second stream (the Gumbel-max trick, an exact draw from
  softmax(dl[t]/T) that evaluates no softmax); this follows the pages'
  requirement that drafts come from the transformed p;
* uniforms: K+2 fp32 draws in [0, 1) from a third stream.
"""

from __future__ import annotations

import torch

from .configs import Workload

DTYPES = {"bf16": torch.bfloat16, "f32": torch.float32}

_MASK64 = (1 << 64) - 1


def _mix(*parts: int) -> int:
    """Deterministic 63-bit seed from integers (splitmix64 finaliser over a sum)."""
    x = 0x243F6A8885A308D3
    for p in parts:
        x = (x + (p & _MASK64) * 0x9E3779B97F4A7C15 + 0x632BE59BD9B4E019) & _MASK64
        x ^= x >> 30
        x = (x * 0xBF58476D1CE4E5B9) & _MASK64
        x ^= x >> 27
        x = (x * 0x94D049BB133111EB) & _MASK64
        x ^= x >> 31
    return x & ((1 << 63) - 1)


def _gen(w: Workload, step: int, b: int, stream: int) -> torch.Generator:
    return torch.Generator().manual_seed(_mix(w.seed, step, b, stream))


def gumbel_max_draw(rows: torch.Tensor, temperature: float, g: torch.Generator) -> torch.Tensor:
    """One index per row of `rows` [n, V], distributed as softmax(rows / T):
    argmax_i(rows_i / T + G_i) with G_i = -log(-log U_i), U_i uniform (fp64)."""
    u = torch.rand(rows.shape, dtype=torch.float64, generator=g)
    gumbel = -torch.log(-torch.log(u))
    return torch.argmax(rows.to(torch.float64) / float(temperature) + gumbel, dim=-1).to(torch.int32)


def make_sequence(w: Workload, step: int, b: int):
    """One sequence: (target [K+1,V], draft [K,V], tokens [K] int32, uniforms [K+2] f32)."""
    dtype = DTYPES[w.dtype]
    g = _gen(w, step, b, 0)
    tl = torch.randn(w.K + 1, w.V, generator=g) * w.target_std
    if w.peaks:
        for r in range(w.K + 1):
            ids = torch.randperm(w.V, generator=g)[: w.peaks]
            tl[r, ids] += w.peak_boost
    dl = tl[: w.K] + torch.randn(w.K, w.V, generator=g) * w.draft_noise_std
    tl = tl.to(dtype)
    dl = dl.to(dtype)

    tokens = gumbel_max_draw(dl, w.temperature, _gen(w, step, b, 1))

    g3 = _gen(w, step, b, 2)
    uniforms = torch.rand(w.K + 2, generator=g3, dtype=torch.float32)
    return tl, dl, tokens, uniforms


def make_inputs(w: Workload, step: int = 0, seqs=None, pin_memory: bool = False):
    """A batch of inputs for workload `w` at verify step `step`.

    `seqs` (optional iterable of sequence indices) generates only those
    sequences, in that order; by default all B. Returns a dict of CPU tensors:
    target [n,K+1,V], draft [n,K,V], tokens [n,K] int32, uniforms [n,K+2] f32,
    and the temperature as a Python float.
    """
    idx = list(range(w.B)) if seqs is None else list(seqs)
    n = len(idx)
    dtype = DTYPES[w.dtype]
    target = torch.empty(n, w.K + 1, w.V, dtype=dtype, pin_memory=pin_memory)
    draft = torch.empty(n, w.K, w.V, dtype=dtype, pin_memory=pin_memory)
    tokens = torch.empty(n, w.K, dtype=torch.int32, pin_memory=pin_memory)
    uniforms = torch.empty(n, w.K + 2, dtype=torch.float32, pin_memory=pin_memory)
    for i, b in enumerate(idx):
        tl, dl, tk, un = make_sequence(w, step, b)
        target[i] = tl
        draft[i] = dl
        tokens[i] = tk
        uniforms[i] = un
    return {
        "target": target,
        "draft": draft,
        "tokens": tokens,
        "uniforms": uniforms,
        "temperature": float(w.temperature),
    }


def topk_draft_tokens(draft: torch.Tensor, top_k: int, temperature: float,
                      g: torch.Generator) -> torch.Tensor:
    """Drafts for top-k decoding: x_t drawn (Gumbel-max) from softmax(dl[t]/T)
    restricted to the top_k largest logits of draft row t (torch.topk's choice
    among equal logits at the cut; any choice is a valid draft)."""
    rows = draft.reshape(-1, draft.shape[-1]).to(torch.float64)
    if top_k < rows.shape[-1]:
        keep = torch.topk(rows, top_k, dim=-1).indices
        masked = torch.full_like(rows, float("-inf"))
        masked.scatter_(-1, keep, rows.gather(-1, keep))
        rows = masked
    return gumbel_max_draw(rows, temperature, g).reshape(draft.shape[:-1])


def make_topk_inputs(w: Workload, top_k: int, step: int = 0, seqs=None, pin_memory: bool = False):
    """`make_inputs` with drafts drawn from the top-k filtered draft rows (a
    fourth per-sequence stream), as a top-k decoding draft model would."""
    inp = make_inputs(w, step=step, seqs=seqs, pin_memory=pin_memory)
    idx = list(range(w.B)) if seqs is None else list(seqs)
    for i, b in enumerate(idx):
        inp["tokens"][i] = topk_draft_tokens(inp["draft"][i], top_k, w.temperature,
                                             _gen(w, step, b, 3))
    return inp


def topp_draft_tokens(draft: torch.Tensor, top_p: float, temperature: float,
                      g: torch.Generator) -> torch.Tensor:
    """Drafts for nucleus decoding: x_t drawn (Gumbel-max) from softmax(dl[t]/T)
    restricted to the shortest prefix of the draft row, in descending order,
    whose probability reaches top_p (torch's sort; any order among equal
    logits gives a valid draft)."""
    rows = draft.reshape(-1, draft.shape[-1]).to(torch.float64)
    if top_p < 1.0:
        q = torch.softmax(rows / float(temperature), dim=-1)
        vals, order = torch.sort(q, dim=-1, descending=True)
        csum = torch.cumsum(vals, dim=-1)
        n_keep = (csum < top_p).sum(dim=-1, keepdim=True) + 1
        pos = torch.arange(rows.shape[-1]).expand_as(order)
        keep = torch.zeros_like(rows, dtype=torch.bool).scatter_(-1, order, pos < n_keep)
        rows = torch.where(keep, rows, torch.full_like(rows, float("-inf")))
    return gumbel_max_draw(rows, temperature, g).reshape(draft.shape[:-1])


def make_topp_inputs(w: Workload, top_p: float, step: int = 0, seqs=None, pin_memory: bool = False):
    """`make_inputs` with drafts drawn from the nucleus filtered draft rows (a
    fifth per-sequence stream), as a nucleus decoding draft model would."""
    inp = make_inputs(w, step=step, seqs=seqs, pin_memory=pin_memory)
    idx = list(range(w.B)) if seqs is None else list(seqs)
    for i, b in enumerate(idx):
        inp["tokens"][i] = topp_draft_tokens(inp["draft"][i], top_p, w.temperature,
                                             _gen(w, step, b, 4))
    return inp


def make_batch(w: Workload, step: int = 0, device="cpu", rows_per_chunk: int = 64):
    """The recipe of `make_inputs`, drawn for the whole batch at once from one
    torch generator on `device` (the device's own generator: on a GPU, torch's
    counter-based Philox), for workloads too large to draw sequence by
    sequence on the host. Same shapes, dtypes and distributions; the values
    differ from `make_inputs`, and are reproducible for a given device type,
    seed and step.

    * target logits N(0, target_std^2) in fp32, plus `peak_boost` on `peaks`
      distinct ids per target row (the ids of the row's `peaks` largest
      uniform draws, a uniformly random subset);
    * draft row t = target row t + N(0, noise^2), t < K;
    * both rounded to the workload dtype (bf16: round to nearest even);
    * drafts by the Gumbel-max trick in fp64, argmax_i(dl[t,i]/T + G_i), an
      exact draw from softmax(dl[t]/T), `rows_per_chunk` draft rows at a time;
    * K+2 fp32 uniforms in [0, 1) per sequence.
    """
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(_mix(w.seed, step, 0x5EED))
    dtype = DTYPES[w.dtype]
    B, K, V = w.B, w.K, w.V
    tl = torch.randn(B, K + 1, V, generator=g, device=dev)
    tl.mul_(w.target_std)
    if w.peaks:
        for r in range(K + 1):
            pick = torch.rand(B, V, generator=g, device=dev)
            ids = torch.topk(pick, w.peaks, dim=-1).indices
            tl[:, r].scatter_add_(-1, ids, torch.full(ids.shape, float(w.peak_boost), device=dev))
            del pick, ids
    noise = torch.randn(B, K, V, generator=g, device=dev)
    noise.mul_(w.draft_noise_std)
    noise.add_(tl[:, :K])
    draft = noise.to(dtype)
    del noise
    target = tl.to(dtype)
    del tl
    rows = draft.view(B * K, V)
    tokens = torch.empty(B * K, dtype=torch.int32, device=dev)
    inv_t = 1.0 / float(w.temperature)
    for r0 in range(0, B * K, rows_per_chunk):
        r1 = min(B * K, r0 + rows_per_chunk)
        u = torch.rand(r1 - r0, V, dtype=torch.float64, generator=g, device=dev)
        gumbel = u.log_().neg_().log_().neg_()
        gumbel.add_(rows[r0:r1].to(torch.float64) * inv_t)
        tokens[r0:r1] = torch.argmax(gumbel, dim=-1).to(torch.int32)
        del u, gumbel
    uniforms = torch.rand(B, K + 2, generator=g, device=dev, dtype=torch.float32)
    return {
        "target": target,
        "draft": draft,
        "tokens": tokens.view(B, K),
        "uniforms": uniforms,
        "temperature": float(w.temperature),
    }


def make_lmhead_inputs(N: int, D: int, V: int, logit_std: float = 3.0, seed: int = 0,
                       device="cpu", none_every: int = 7):
    """Hidden states h [N, D] ~ N(0, 1) and projection weights W [V, D] ~
    N(0, logit_std^2 / D), both rounded to bf16, so that the logits h W^T have
    about `logit_std` spread; one token per row, uniform over [0, V), with
    every `none_every`-th row given -1 (no token). One torch generator on
    `device`."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(_mix(seed, N, D, V))
    h = torch.randn(N, D, generator=g, device=dev).to(torch.bfloat16)
    w = (torch.randn(V, D, generator=g, device=dev) * (logit_std / D ** 0.5)).to(torch.bfloat16)
    tok = torch.randint(0, V, (N,), generator=g, device=dev, dtype=torch.int64).to(torch.int32)
    if none_every:
        tok[::none_every] = -1
    return {"hidden": h, "weight": w, "tokens": tok}
