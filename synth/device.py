"""Device-resident decode problems built from the seeded draws.

Uploads the drawn weights, queries and sequences with torch (device memory
only) and fills the paged cache through the library's own public calls
(mla_absorb_weights, mla_cache_append).  No attention arithmetic here.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .workloads import (D_C, D_NOPE, D_R, D_V, PAGE, Workload, gen_queries, gen_seqlens, gen_sequence,
                        gen_weights, make_page_table)


@dataclass
class Problem:
    H: int
    seqlens: np.ndarray          # int32 [B]
    seed: int
    dist: str = "rmsnorm"
    fmt: str = "bf16"
    paged: bool = True
    scale: float = 1.0 / (D_NOPE + D_R) ** 0.5
    spare_pages: int = 0
    wkv: np.ndarray = field(default=None, repr=False)       # bf16 bits [H*256, 512]
    q_nope: np.ndarray = field(default=None, repr=False)    # bf16 bits [B, H, 128]
    q_pe: np.ndarray = field(default=None, repr=False)      # bf16 bits [B, H, 64]
    page_table: np.ndarray = field(default=None, repr=False)
    num_pages: int = 0

    @property
    def B(self) -> int:
        return len(self.seqlens)

    @property
    def max_pages(self) -> int:
        return self.page_table.shape[1]

    def sequence(self, b: int, start: int = 0, n: int | None = None):
        """bf16 bits (c_kv [n,512], k_pe [n,64]) of row b, tokens [start, start+n)."""
        n = int(self.seqlens[b]) - start if n is None else n
        return gen_sequence(self.seed, b, n, self.dist, start=start)

    @property
    def cache_tokens(self) -> int:
        return int(np.sum(self.seqlens))


def make_problem(H: int, seqlens, seed: int, *, paged: bool = True, dist: str = "rmsnorm", fmt: str = "bf16",
                 spare_pages: int = 0) -> Problem:
    seqlens = np.asarray(seqlens, dtype=np.int32)
    p = Problem(H=H, seqlens=seqlens, seed=seed, dist=dist, fmt=fmt, paged=paged, spare_pages=spare_pages)
    p.wkv = gen_weights(H, seed)
    p.q_nope, p.q_pe = gen_queries(H, seqlens, seed)
    p.page_table, p.num_pages = make_page_table(seqlens, seed, paged, spare_pages)
    return p


def problem_from_workload(w: Workload, fmt: str | None = None) -> Problem:
    return make_problem(w.H, gen_seqlens(w), w.seed, paged=w.paged, dist=w.dist, fmt=fmt or w.fmts[0])


def bits_to_device(bits: np.ndarray, device="cuda"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


class DeviceDecode:
    """A problem resident on the GPU: absorbed weights, filled paged cache,
    queries, lengths, workspace and output buffer."""

    def __init__(self, prob: Problem, device="cuda", prefill: int | None = None, rows_per_append: int = 8):
        import torch
        import mla_absorbed_latent_gb300 as mla
        self.mla, self.torch, self.prob, self.device = mla, torch, prob, device
        H, B = prob.H, prob.B
        self.wkv = bits_to_device(prob.wkv, device)
        self.W_UK = torch.empty((H, D_C, D_NOPE), dtype=torch.bfloat16, device=device)
        self.W_UV = torch.empty((H, D_V, D_C), dtype=torch.bfloat16, device=device)
        mla.mla_absorb_weights(self.wkv, H, self.W_UK, self.W_UV)
        self.page_bytes = mla.mla_cache_page_bytes(prob.fmt)
        self.pool = torch.zeros(prob.num_pages * self.page_bytes, dtype=torch.uint8, device=device)
        self.cache = mla.cache_struct(prob.fmt, prob.num_pages, self.pool)
        self.page_table = torch.from_numpy(prob.page_table).to(device)
        self.seqlens = torch.from_numpy(prob.seqlens.astype(np.int32)).to(device)
        self.q_nope = bits_to_device(prob.q_nope, device)
        self.q_pe = bits_to_device(prob.q_pe, device)
        self.ws_bytes = mla.mla_decode_workspace_bytes(B, H)
        self.workspace = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=device)
        self.out = torch.empty((B, H, D_V), dtype=torch.bfloat16, device=device)
        self.fill(prefill, rows_per_append)

    def append(self, rows, start: int, n: int) -> None:
        """Append tokens [start, start+n) of the listed rows (all the same n)."""
        torch, mla, prob = self.torch, self.mla, self.prob
        cs, ps = zip(*(prob.sequence(b, start, n) for b in rows))
        c = bits_to_device(np.stack(cs), self.device)
        p = bits_to_device(np.stack(ps), self.device)
        pt = self.page_table[list(rows)].contiguous()
        pos = torch.full((len(rows),), start, dtype=torch.int32, device=self.device)
        mla.mla_cache_append(self.cache, c, p, pt, prob.max_pages, pos, len(rows), n)

    def fill(self, prefill: int | None = None, rows_per_append: int = 8) -> None:
        prob = self.prob
        by_len: dict[int, list[int]] = {}
        for b, n in enumerate(prob.seqlens.tolist()):
            if n > 0:
                by_len.setdefault(int(n), []).append(b)
        for n, rows in by_len.items():
            for i in range(0, len(rows), rows_per_append):
                chunk = rows[i:i + rows_per_append]
                if prefill is not None and 0 < prefill < n:
                    self.append(chunk, 0, prefill)
                    self.append(chunk, prefill, n - prefill)
                else:
                    self.append(chunk, 0, n)
        self.torch.cuda.synchronize()

    def decode(self, stream=None):
        p = self.prob
        self.mla.mla_decode(self.q_nope, self.q_pe, self.W_UK, self.W_UV, p.H, self.cache, self.page_table,
                            p.max_pages, self.seqlens, p.B, p.scale, self.workspace, self.ws_bytes, self.out,
                            stream)
        return self.out

    def decode_steps(self, o_lat=None, stream=None):
        p, m = self.prob, self.mla
        m.mla_decode_plan(p.H, p.fmt, self.seqlens, p.B, p.max_pages, self.workspace, self.ws_bytes, stream)
        m.mla_decode_absorb_q(self.q_nope, self.q_pe, self.W_UK, p.H, p.B, self.workspace, self.ws_bytes, stream)
        m.mla_decode_attend(p.H, self.cache, self.page_table, p.max_pages, self.seqlens, p.B, p.scale,
                            self.workspace, self.ws_bytes, stream)
        m.mla_decode_combine(self.W_UV, p.H, p.B, self.workspace, self.ws_bytes, self.out, o_lat, stream)
        return self.out
