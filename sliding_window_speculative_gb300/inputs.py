"""Seeded synthetic inputs for sliding-window verify attention.

This module only draws and lays out inputs; it holds none of the method's
arithmetic.  Both the CUDA path (tests, bench) and the fp64 oracle checks
take their inputs from here.

Workloads (single-stream Gemma-style serving: 8 query / 2 KV heads, head
dim 256, draft block of 1 committed + 7 drafted tokens, window 188; see
"The Fast Gemma Challenge: our verified-SOTA recipe, in full", manifest keys
SLIDING_WINDOW, SPECULATIVE_CONFIG num_speculative_tokens=7,
SPLITKV_VERIFY_MAX_Q=64, MAX_MODEL_LEN=4096):

  tiny           B=1, Hq/Hkv 2/1, D 64, context 40, W 16, q_len 1 (p=39) or 8 (p=32..39)
  single_stream  B=1, 8/2, D 256, context 4096, W 188, q_len 8, 1% of K entries x8
  window_vs_full single_stream's tensors, q_len 1 (its last draft row), W 188 or 4096
  batched        B=64, context ~ U[200, 4096], 8/2, D 256, W 188, q_len 8
  stress         B=512, context ~ U[1024, 32768], 8/2, D 256, W in {188,512,1024},
                 q_len in {1,8,64}, 1% of K entries x8, cache length 32768

Values are bf16 N(0, 1).  "1% of key entries x8" is an elementwise
Bernoulli(0.01) mask on K, multiplied by 8 before the bf16 cast (exact).
Context lengths are integers drawn uniformly, inclusive, from a CPU
generator seeded with `seed`; q_pos = seq_len - q_len (tiny q_len 1: the last
token; window_vs_full: the last token).

Cache rows that no query may see are filled with poison (K = 0, V = 1e4 by
default, or NaN), and the cache tensors are views into larger buffers whose
guard bands before and after hold the same poison, so a read outside the
window shows up as a large error.
"""
from dataclasses import dataclass, field
import math

import torch

POISON_K = 0.0
POISON_V = 1.0e4


@dataclass
class Case:
    name: str
    q: torch.Tensor            # bf16 [B, q_len, Hq, D]
    k_cache: torch.Tensor      # bf16 [B, Hkv, max_len, D] (a view inside k_buf)
    v_cache: torch.Tensor
    seq_lens: torch.Tensor     # int32 [B]
    q_pos: torch.Tensor        # int32 [B]
    window: int
    scale: float
    seq_lens_host: list = field(default_factory=list)
    q_pos_host: list = field(default_factory=list)
    k_buf: torch.Tensor = None  # whole buffer including guard bands
    v_buf: torch.Tensor = None

    @property
    def dims(self):
        B, q_len, Hq, D = self.q.shape
        Hkv, L = self.k_cache.shape[1], self.k_cache.shape[2]
        return dict(batch=B, q_len=q_len, num_q_heads=Hq, num_kv_heads=Hkv,
                    head_dim=D, max_len=L)

    def span(self, margin=0):
        """Per sequence, the absolute rows [start, seq_len) that a query may
        see, widened by `margin` rows before the first one."""
        out = []
        for sl, qp in zip(self.seq_lens_host, self.q_pos_host):
            start = max(0, qp - self.window + 1 - margin)
            out.append((start, sl))
        return out


def _guarded(shape, guard_rows, device, fill):
    """A [B, H, L, D] bf16 view inside a flat buffer with `guard_rows` rows
    (of D) of `fill` before and after."""
    B, H, L, D = shape
    n = B * H * L * D + 2 * guard_rows * D
    buf = torch.full((n,), fill, dtype=torch.bfloat16, device=device)
    view = buf[guard_rows * D: guard_rows * D + B * H * L * D].view(B, H, L, D)
    return buf, view


def _randn_bf16(shape, gen, device, outliers):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if outliers:
        mask = torch.rand(shape, generator=gen, device=device) < 0.01
        x = torch.where(mask, x * 8.0, x)
    return x.to(torch.bfloat16)


def make_case(name, B, Hq, Hkv, D, q_len, window, seq_lens, max_len, q_pos=None,
              seed=0, outliers=False, device="cpu", gen_device="cpu", fill="full",
              margin=64, poison="finite", guard_rows=64, q=None, kv=None):
    """Draw one workload.

    fill="full":   every cache row below seq_len is N(0,1); rows >= seq_len poison.
    fill="window": only rows [max(0, q_pos-W+1-margin), seq_len) are N(0,1);
                   everything else is poison (cheap for long caches).
    poison:        "finite" (K=0, V=1e4) or "nan".
    q / kv:        reuse given tensors instead of drawing new ones.
    """
    seq_lens = [int(s) for s in seq_lens]
    if q_pos is None:
        q_pos = [s - q_len for s in seq_lens]
    q_pos = [int(p) for p in q_pos]
    pk, pv = (POISON_K, POISON_V) if poison == "finite" else (float("nan"), float("nan"))
    gen = torch.Generator(device=gen_device)
    gen.manual_seed(seed)
    if q is None:
        q = _randn_bf16((B, q_len, Hq, D), gen, gen_device, False)
    q = q.to(device).contiguous()
    if kv is not None:
        k_buf, v_buf, k_cache, v_cache = kv
    else:
        k_buf, k_cache = _guarded((B, Hkv, max_len, D), guard_rows, device, pk)
        v_buf, v_cache = _guarded((B, Hkv, max_len, D), guard_rows, device, pv)
        if fill == "full":
            L = max(seq_lens)
            k = _randn_bf16((B, Hkv, L, D), gen, gen_device, outliers).to(device)
            v = _randn_bf16((B, Hkv, L, D), gen, gen_device, False).to(device)
            for b, sl in enumerate(seq_lens):
                k_cache[b, :, :sl] = k[b, :, :sl]
                v_cache[b, :, :sl] = v[b, :, :sl]
            del k, v
        elif fill == "window":
            S = max(sl - max(0, qp - window + 1 - margin) for sl, qp in zip(seq_lens, q_pos))
            k = _randn_bf16((B, Hkv, S, D), gen, gen_device, outliers).to(device)
            v = _randn_bf16((B, Hkv, S, D), gen, gen_device, False).to(device)
            for b, (sl, qp) in enumerate(zip(seq_lens, q_pos)):
                st = max(0, qp - window + 1 - margin)
                k_cache[b, :, st:sl] = k[b, :, :sl - st]
                v_cache[b, :, st:sl] = v[b, :, :sl - st]
            del k, v
        else:
            raise ValueError(fill)
        if poison == "nan":
            # rows before the first one any query can see are poison as well
            for b, (sl, qp) in enumerate(zip(seq_lens, q_pos)):
                st = max(0, qp - window + 1)
                k_cache[b, :, :st] = pk
                v_cache[b, :, :st] = pv
    return Case(name=name, q=q, k_cache=k_cache, v_cache=v_cache,
                seq_lens=torch.tensor(seq_lens, dtype=torch.int32, device=device),
                q_pos=torch.tensor(q_pos, dtype=torch.int32, device=device),
                window=int(window), scale=1.0 / math.sqrt(D),
                seq_lens_host=seq_lens, q_pos_host=q_pos, k_buf=k_buf, v_buf=v_buf)


def context_lengths(n, lo, hi, seed=0):
    """n integers uniform in [lo, hi], inclusive, from a CPU generator."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


# ---------------------------------------------------------------- named cases

def tiny(q_len, device="cpu", **kw):
    q_pos = 39 if q_len == 1 else 40 - q_len
    return make_case(f"tiny_q{q_len}", 1, 2, 1, 64, q_len, 16, [40], 40, q_pos=[q_pos],
                     device=device, **kw)


def single_stream(device="cpu", **kw):
    return make_case("single_stream", 1, 8, 2, 256, 8, 188, [4096], 4096, outliers=True,
                     device=device, **kw)


def window_vs_full(window, device="cpu", base=None, **kw):
    """single_stream's tensors, q_len 1 = its last draft row (position 4095)."""
    base = base or single_stream(device=device, **kw)
    q1 = base.q[:, -1:].contiguous()
    return make_case(f"window_vs_full_w{window}", 1, 8, 2, 256, 1, window, [4096], 4096,
                     q_pos=[4095], device=device, q=q1,
                     kv=(base.k_buf, base.v_buf, base.k_cache, base.v_cache), **kw)


def batched(device="cpu", gen_device=None, **kw):
    lens = context_lengths(64, 200, 4096)
    return make_case("batched", 64, 8, 2, 256, 8, 188, lens, 4096, device=device,
                     gen_device=gen_device or device, fill="window", **kw)


def prefill(q_len, window=188, batch=1, device="cuda", max_len=4096, gen_device=None, **kw):
    """Sliding-window prefill chunks: `batch` sequences whose last q_len
    positions form the chunk (contexts U[q_len, max_len], q_pos = seq_len -
    q_len), single_stream's heads and head_dim."""
    lens = context_lengths(batch, q_len, max_len)
    return make_case(f"prefill_q{q_len}", batch, 8, 2, 256, q_len, window, lens, max_len,
                     outliers=True, device=device, gen_device=gen_device or device,
                     fill="window", **kw)


def stress(window, q_len, device="cuda", batch=512, max_len=32768, gen_device=None, **kw):
    lens = context_lengths(batch, 1024, max_len)
    return make_case(f"stress_w{window}_q{q_len}", batch, 8, 2, 256, q_len, window, lens,
                     max_len, outliers=True, device=device,
                     gen_device=gen_device or device, fill="window", **kw)

