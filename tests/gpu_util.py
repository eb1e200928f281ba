"""Helpers for the GPU parity tests: run a workload through the C ABI and
build the oracle's view of the same sequence from the same seeded inputs."""

from __future__ import annotations

import numpy as np

import oracle
from workloads import synthetic as syn

MAX_ABS = 2e-3
REL_L2 = 1e-3

_TOKEN_CACHE = {}


def cached_tokens(w: syn.Workload, b: int, scales):
    """Seeded tokens, shared by workloads with the same seed, lengths and steps."""
    key = (w.seed, w.length_kind, w.length_args, w.batch, w.steps, b)
    if key not in _TOKEN_CACHE:
        if len(_TOKEN_CACHE) > 16:
            _TOKEN_CACHE.clear()
        _TOKEN_CACHE[key] = syn.sequence_tokens(w, b, scales=scales)
    return _TOKEN_CACHE[key]


def to_dev(a, dtype, dev="cuda"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(dev).view(dtype)


GUARD_BYTES = 4096
GUARD_FILL = 0xA5


class Guards:
    """Device buffers with guard bytes before and after them: a kernel that
    writes outside a buffer it is given changes a guard."""

    def __init__(self, torch, dev):
        self.torch = torch
        self.dev = dev
        self.regions = []

    def alloc(self, shape, dtype, what):
        torch = self.torch
        n = int(np.prod(shape)) * torch.empty(0, dtype=dtype).element_size()
        n16 = (n + 15) // 16 * 16
        full = torch.full((GUARD_BYTES + n16 + GUARD_BYTES,), GUARD_FILL, dtype=torch.uint8,
                          device=self.dev)
        self.regions.append((what, full, n))
        return full[GUARD_BYTES:GUARD_BYTES + n].view(dtype).view(*shape)

    def check(self):
        for what, full, n in self.regions:
            head = full[:GUARD_BYTES]
            tail = full[GUARD_BYTES + n:]
            assert bool((head == GUARD_FILL).all()), f"guard bytes before {what} overwritten"
            assert bool((tail == GUARD_FILL).all()), f"guard bytes after {what} overwritten"


class GpuRun:
    """One workload on the GPU: prefill, then ``steps`` writer + decode steps.
    The page pool, bf16 buffers, outputs and workspace sit between guard bytes
    (``guards.check()``)."""

    def __init__(self, w: syn.Workload, dev: str = "cuda", rotate: bool = False):
        import torch
        import bit_mla_kv_lowbit_gb300 as pkg
        self.torch = torch
        self.w = w
        self.dev = dev
        self.lens = syn.sequence_lengths(w)
        self.table, self.npages = syn.make_paging(w)
        self.rotate = rotate
        self.cache = pkg.PagedCache(w.content_bits, w.rope_bits, self.table, self.npages, dev,
                                    rotate=rotate)
        self.guards = Guards(torch, dev)
        c = self.cache
        c.pool = self.guards.alloc(tuple(c.pool.shape), torch.uint8, "page pool")
        c.pool.zero_()
        if c.sink is not None:
            c.sink = self.guards.alloc(tuple(c.sink.shape), torch.bfloat16, "sink buffer")
            c.recent = self.guards.alloc(tuple(c.recent.shape), torch.bfloat16, "recent buffer")
            c.sink.zero_()
            c.recent.zero_()
        self.out = self.guards.alloc((w.batch, w.heads, 512), torch.float32, "output")
        self.lse = self.guards.alloc((w.batch, w.heads), torch.float32, "lse")
        self._ws = None
        self.scales = syn.channel_scales(w)
        self.tokens = {}
        self.step = -1

    def workspace(self, lens_host):
        """Guarded workspace for this run's row count, grown to the plan's size."""
        import bit_mla_kv_lowbit_gb300 as pkg
        _, _, nbytes = pkg.decode_plan(self.cache.layout, self.w.heads, lens_host)
        if self._ws is None or self._ws.numel() < nbytes:
            self._ws = self.guards.alloc((max(int(nbytes), 16),), self.torch.uint8, "workspace")
        return self._ws

    def seq_tokens(self, b):
        if b not in self.tokens:
            self.tokens[b] = cached_tokens(self.w, b, self.scales)
        return self.tokens[b]

    def prefill(self, keep_tokens=True):
        """Write positions 0..L_b-2 of every sequence (one call per sequence)."""
        torch = self.torch
        for b in range(self.w.batch):
            n = int(self.lens[b]) - 1
            if n <= 0:
                continue
            ckv, kr = self.seq_tokens(b)
            self.cache.write(to_dev(ckv[:n], torch.bfloat16, self.dev),
                             to_dev(kr[:n], torch.bfloat16, self.dev),
                             torch.arange(n, dtype=torch.int32, device=self.dev),
                             seq_idx=torch.full((n,), b, dtype=torch.int32, device=self.dev),
                             seq_lens_after=to_dev((self.lens - 1).astype(np.int32), torch.int32,
                                                   self.dev))
            if not keep_tokens:
                self.tokens.pop(b, None)

    def step_inputs(self, s):
        """New token of each sequence at step s and the queries of step s."""
        B = self.w.batch
        ckv = np.empty((B, 512), np.uint16)
        kr = np.empty((B, 64), np.uint16)
        for b in range(B):
            c, k = self.seq_tokens(b)
            p = int(self.lens[b]) - 1 + s
            ckv[b], kr[b] = c[p], k[p]
        q = np.stack([syn.queries(self.w, b)[s] for b in range(B)])
        return ckv, kr, q

    def run_step(self, s, lse=False, fused=False):
        """Writer for step s then decode over lens + s (one mla_lowbit_write_decode
        call when ``fused``).  Returns (out, lse)."""
        torch = self.torch
        ckv, kr, q = self.step_inputs(s)
        pos = (self.lens - 1 + s).astype(np.int32)
        lens_now = (self.lens + s).astype(np.int32)
        lse_t = self.lse if lse else None
        ws = self.workspace([int(x) for x in lens_now])
        if fused:
            out = self.cache.write_decode(
                to_dev(ckv, torch.bfloat16, self.dev), to_dev(kr, torch.bfloat16, self.dev),
                to_dev(q, torch.bfloat16, self.dev), to_dev(lens_now, torch.int32, self.dev),
                lens_now, self.w.softmax_scale, out=self.out, lse=lse_t, workspace=ws)
            torch.cuda.synchronize()
            self.guards.check()
            self.step = s
            return out.cpu().numpy(), (lse_t.cpu().numpy() if lse else None)
        self.cache.write(to_dev(ckv, torch.bfloat16, self.dev), to_dev(kr, torch.bfloat16, self.dev),
                         to_dev(pos, torch.int32, self.dev),
                         seq_lens_after=to_dev(lens_now, torch.int32, self.dev))
        out = self.cache.decode(to_dev(q, torch.bfloat16, self.dev),
                                to_dev(lens_now, torch.int32, self.dev), lens_now,
                                self.w.softmax_scale, out=self.out, lse=lse_t, workspace=ws)
        torch.cuda.synchronize()
        self.guards.check()
        self.step = s
        return out.cpu().numpy(), (lse_t.cpu().numpy() if lse else None)

    def pages_of(self, b, L):
        n = (L + 63) // 64
        return self.table[b, :n]


def oracle_model(run: GpuRun, b: int, s: int):
    """Oracle cache model holding sequence b after step s (its own writer)."""
    w = run.w
    lay = oracle.Layout(w.content_bits, w.rope_bits, rotate=run.rotate)
    model = oracle.PagedCacheModel(lay, run.npages, run.table)
    L = int(run.lens[b]) + s
    ckv, kr = run.seq_tokens(b)
    # prefill in one call, then the step tokens one by one (the same ring rule)
    n0 = int(run.lens[b]) - 1
    lens_after = np.zeros(w.batch, np.int64)
    if n0 > 0:
        lens_after[b] = n0
        model.write(np.full(n0, b), np.arange(n0), ckv[:n0], kr[:n0], lens_after)
    for p in range(n0, L):
        lens_after[b] = p + 1
        model.write([b], [p], ckv[p:p + 1], kr[p:p + 1], lens_after)
    return model, L


def check_attention(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref).max() if ref.size else 0.0
    nrm = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / nrm if nrm > 0 else np.linalg.norm(got - ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert err <= MAX_ABS and rel <= REL_L2, f"{what}: max-abs {err:.3e}, rel-L2 {rel:.3e}"
    return err, rel
