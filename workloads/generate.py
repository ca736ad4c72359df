"""Seeded generators for the synthetic verification inputs.

Two backends draw the logits: ``numpy`` (host, bit-reproducible on any machine; used for the small
workloads and the oracle's tests) and ``torch`` (the device generator of the current CUDA device,
used for the multi-GB workloads so that a benchmark does not spend minutes on host-side random
numbers). Per-row scalars (draft lengths, temperatures, the greedy subset, uniforms) always come from
numpy, so the verified-position count of every workload is fixed by its seed alone.

Draft tokens are drawn from the draft distribution by the Gumbel-max method (argmax of
z_d / T + Gumbel noise) -- an exact sample from softmax(z_d / T) that needs no normalisation.
Greedy rows take the draft argmax (a greedy drafter). The drafting step sits upstream of
verification; nothing here computes a verification quantity.

Padding is poisoned so that a kernel that reads it fails parity: target rows past position gamma_b,
draft rows at or past gamma_b and every draft row of a greedy row hold NaN, and draft tokens at or
past gamma_b hold -1.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .configs import Config, get_config

ELEM_BYTES = {"f32": 4, "bf16": 2}


def bf16_round(x):
    """Round float32 values to the nearest bfloat16 (ties to even), returned as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    r = ((bits + 0x7FFF + ((bits >> 16) & 1)) >> 16) << 16
    out = r.astype(np.uint32).view(np.float32)
    return np.where(np.isnan(x), np.float32(np.nan), out)


def bf16_bits_to_f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _row_params(cfg: Config, seed: int):
    """Per-row scalars: draft_len, temperature, sigma, uniforms, greedy mask, Zipf permutation."""
    B, G, V = cfg.B, cfg.gamma_max, cfg.V
    uniforms = np.random.default_rng(seed).random((B, G + 2), dtype=np.float32)
    ss = np.random.SeedSequence(seed)
    r_rows, r_perm = (np.random.default_rng(s) for s in ss.spawn(2))
    if cfg.ragged:
        draft_len = r_rows.integers(1, G + 1, size=B).astype(np.int32)
    else:
        draft_len = np.full(B, G, dtype=np.int32)
    if isinstance(cfg.temperature, tuple):
        temperature = r_rows.uniform(*cfg.temperature, size=B).astype(np.float32)
    else:
        temperature = np.full(B, cfg.temperature, dtype=np.float32)
    if isinstance(cfg.sigma, tuple):
        sigma = r_rows.uniform(*cfg.sigma, size=B).astype(np.float32)
    else:
        sigma = np.full(B, cfg.sigma, dtype=np.float32)
    greedy = np.zeros(B, dtype=bool)
    if cfg.greedy == "odd":
        greedy[1::2] = True
    elif cfg.greedy.startswith("frac:"):
        n = int(round(float(cfg.greedy[5:]) * B))
        greedy[r_rows.permutation(B)[:n]] = True
    temperature[greedy] = 0.0
    if cfg.zipf:
        rank = 1.0 + r_perm.permutation(V).astype(np.float64)
        bias = (-cfg.zipf * np.log(rank)).astype(np.float32)
    else:
        bias = np.zeros(V, dtype=np.float32)
    return draft_len, temperature, sigma, uniforms, greedy, bias


@dataclass
class Workload:
    cfg: Config
    backend: str
    target_logits: object      # [B, G+1, V]: numpy float32 (values exact in cfg.dtype) or torch tensor
    draft_logits: object       # [B, G, V]
    draft_tokens: np.ndarray   # [B, G] int32
    draft_len: np.ndarray      # [B] int32
    temperature: np.ndarray    # [B] float32, 0 = greedy
    uniforms: np.ndarray       # [B, G+2] float32 in [0, 1)

    @property
    def B(self):
        return self.cfg.B

    @property
    def G(self):
        return self.cfg.gamma_max

    @property
    def V(self):
        return self.cfg.V

    @property
    def elem_bytes(self):
        return ELEM_BYTES[self.cfg.dtype]

    def positions(self) -> int:
        """Verified positions: sum over rows of (gamma_b + 1)."""
        return int(np.sum(self.draft_len.astype(np.int64) + 1))

    def algorithmic_bytes(self, onehot: bool = False) -> int:
        """Logit bytes the method must read once: (2 gamma_b + 1) rows for a sampled row, gamma_b + 1
        target rows for a greedy row (and for every row when the drafts are one-hot: no draft
        logits exist), plus the per-row scalars, tokens, uniforms and outputs."""
        g = self.draft_len.astype(np.int64)
        greedy = (self.temperature == 0) | onehot
        rows = np.where(greedy, g + 1, 2 * g + 1)
        logit = int(np.sum(rows)) * self.V * self.elem_bytes
        G = self.G
        small = self.B * (4 * G + 4 * (G + 2) + 8 + 4 * (G + 1) + 4 + 4 * G)
        return logit + small

    def host_rows(self, b):
        """(target [G+1, V], draft [G, V]) of row b as float32 numpy arrays (exact stored values)."""
        if self.backend == "numpy":
            return self.target_logits[b], self.draft_logits[b]
        return (self.target_logits[b].float().cpu().numpy(),
                self.draft_logits[b].float().cpu().numpy())

    def device_tensors(self, device="cuda"):
        """Inputs as torch tensors on ``device`` (logits in the storage dtype)."""
        import torch
        tdt = torch.bfloat16 if self.cfg.dtype == "bf16" else torch.float32
        if self.backend == "numpy":
            zt = torch.from_numpy(self.target_logits).to(device=device).to(tdt)
            zd = torch.from_numpy(self.draft_logits).to(device=device).to(tdt)
        else:
            zt, zd = self.target_logits.to(device), self.draft_logits.to(device)
        return dict(
            target_logits=zt.contiguous(), draft_logits=zd.contiguous(),
            draft_tokens=torch.from_numpy(self.draft_tokens).to(device),
            draft_len=torch.from_numpy(self.draft_len).to(device),
            temperature=torch.from_numpy(self.temperature).to(device),
            uniforms=torch.from_numpy(self.uniforms).to(device),
        )


def filter_params(B, seed):
    """Per-row sampling filters of a serving batch: top_k [B] int32 drawn from {0 (off), 20, 50, 100}
    and top_p [B] float32 from {1.0 (off), 0.9, 0.95}, seeded."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 7]))
    top_k = rng.choice(np.array([0, 20, 50, 100], dtype=np.int32), size=B).astype(np.int32)
    top_p = rng.choice(np.array([1.0, 0.9, 0.95], dtype=np.float32), size=B).astype(np.float32)
    return top_k, top_p


def _gumbel_argmax_np(zd_rows, T, rng):
    g = rng.random(zd_rows.shape)
    g = -np.log(-np.log(np.clip(g, 1e-300, None)))
    return np.argmax(zd_rows.astype(np.float64) / np.float64(T) + g, axis=-1)


def make_workload(key, seed=None, backend="numpy", device=None, poison=True, draft_sampler=None,
                  chunk_rows=32) -> Workload:
    """Build workload ``key`` (1..5 or a name) with the given seed (default: the config's seed).

    draft_sampler(draft_logits [B, G, V] float32, temperature [B], uniforms [B, G]) -> [B, G] int,
    if given, replaces the Gumbel-max draft sampler (the tests pass the oracle's inverse-CDF sampler
    for the tiny fp32 workload).
    """
    cfg = get_config(key) if not isinstance(key, Config) else key
    seed = cfg.seed if seed is None else seed
    B, G, V = cfg.B, cfg.gamma_max, cfg.V
    draft_len, temperature, sigma, uniforms, greedy, bias = _row_params(cfg, seed)
    ss = np.random.SeedSequence([seed, 1])
    s_logits, s_draw = ss.spawn(2)

    if backend == "numpy":
        rng = np.random.default_rng(s_logits)
        zt = np.empty((B, G + 1, V), dtype=np.float32)
        zd = np.empty((B, G, V), dtype=np.float32)
        for b in range(B):
            t = rng.standard_normal((G + 1, V), dtype=np.float32) * np.float32(cfg.target_std) + bias
            n = rng.standard_normal((G, V), dtype=np.float32)
            if cfg.draft == "scaled":
                d = np.float32(0.9) * t[:G] + np.float32(sigma[b]) * n
            else:
                d = t[:G] + np.float32(sigma[b]) * n
            if cfg.dtype == "bf16":
                t, d = bf16_round(t), bf16_round(d)
            zt[b], zd[b] = t, d
        rng_d = np.random.default_rng(s_draw)
        if draft_sampler is not None:
            draw_u = rng_d.random((B, G), dtype=np.float32)
            tokens = np.asarray(draft_sampler(zd, temperature, draw_u), dtype=np.int32)
        else:
            tokens = np.zeros((B, G), dtype=np.int32)
            for b in range(B):
                if greedy[b]:
                    tokens[b] = np.argmax(zd[b], axis=-1)
                else:
                    tokens[b] = _gumbel_argmax_np(zd[b], temperature[b], rng_d)
        if poison:
            for b in range(B):
                g = int(draft_len[b])
                zt[b, g + 1:] = np.nan
                zd[b, g:] = np.nan
                if greedy[b]:
                    zd[b] = np.nan
                tokens[b, g:] = -1
        return Workload(cfg, "numpy", zt, zd, tokens, draft_len, temperature, uniforms)

    if backend != "torch":
        raise ValueError(backend)
    import torch
    device = device or "cuda"
    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    gen = torch.Generator(device=device)
    gen.manual_seed(int(s_logits.generate_state(1)[0]))
    bias_t = torch.from_numpy(bias).to(device)
    zt = torch.empty((B, G + 1, V), dtype=tdt, device=device)
    zd = torch.empty((B, G, V), dtype=tdt, device=device)
    tokens = torch.empty((B, G), dtype=torch.int64, device=device)
    temp_t = torch.from_numpy(temperature).to(device)
    sig_t = torch.from_numpy(sigma).to(device)
    greedy_t = torch.from_numpy(greedy).to(device)
    for b0 in range(0, B, chunk_rows):
        nb = min(chunk_rows, B - b0)
        t = torch.randn((nb, G + 1, V), generator=gen, device=device) * cfg.target_std + bias_t
        n = torch.randn((nb, G, V), generator=gen, device=device)
        s = sig_t[b0:b0 + nb, None, None]
        d = (0.9 * t[:, :G] + s * n) if cfg.draft == "scaled" else (t[:, :G] + s * n)
        zt[b0:b0 + nb] = t.to(tdt)
        zd[b0:b0 + nb] = d.to(tdt)
        del t, n, d
        ds = zd[b0:b0 + nb].float()
        u = torch.rand((nb, G, V), generator=gen, device=device).clamp_(min=1e-30)
        T = temp_t[b0:b0 + nb].clamp(min=1e-30)[:, None, None]
        sampled = torch.argmax(ds / T - torch.log(-torch.log(u)), dim=-1)
        greedy_tok = torch.argmax(ds, dim=-1)
        tokens[b0:b0 + nb] = torch.where(greedy_t[b0:b0 + nb, None], greedy_tok, sampled)
        del ds, u
    tokens = tokens.to(torch.int32).cpu().numpy()
    if poison:
        for b in range(B):
            g = int(draft_len[b])
            if g + 1 <= G:
                zt[b, g + 1:] = float("nan")
            if g < G:
                zd[b, g:] = float("nan")
            if greedy[b]:
                zd[b] = float("nan")
            tokens[b, g:] = -1
    torch.cuda.synchronize(device)
    return Workload(cfg, "torch", zt, zd, tokens, draft_len, temperature, uniforms)
