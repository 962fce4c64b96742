"""GPU parity at the full sizes the bench times for the rows beyond the plain
verify call, with the plan the library picks (no forced kernel): the oracle
checks a seeded subset of sequences of each launch.

- prefill chunks of 512 tokens for 64 sequences (prefill_q512_b64);
- the bandwidth-stress batch (512 sequences, cache 32768) on a paged cache
  of 16-row pages, the pool shuffled as in the bench;
- the fused KV append on the bandwidth-stress batch: the sampled sequences'
  new cache rows bit for bit, and their outputs;
- the plain verify call on the bandwidth-stress batch at draft lengths 1 and
  8 for every window: all 512 sequences, not a sample (the oracle needs a
  few seconds per case: each sequence reads at most W + 7 keys); at draft
  length 64 a seeded subset of 64 sequences.
"""
import numpy as np
import pytest
import torch

import oracle
from sliding_window_speculative_gb300 import inputs
from tests.helpers import compare, oracle_reference, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sliding_window_speculative_gb300 import build
    build.build()
    yield


def _sample(case, n, seed):
    rng = np.random.default_rng(seed)
    B = case.q.shape[0]
    seqs = set(rng.choice(B, size=min(n, B), replace=False).tolist())
    seqs.add(int(np.argmin(case.seq_lens_host)))
    seqs.add(int(np.argmax(case.seq_lens_host)))
    return sorted(seqs)


def test_prefill_full_size_sampled():
    case = inputs.prefill(512, batch=64, device="cuda")
    out, lse = run_gpu(case)
    seqs = _sample(case, 6, 51)
    ref_o, ref_l = oracle_reference(case, seqs)
    compare(out[seqs], lse[seqs], ref_o, ref_l, "prefill_q512_b64")
    del case
    torch.cuda.empty_cache()


def test_paged_stress_full_size_sampled():
    from sliding_window_speculative_gb300 import swa_verify_attn_paged
    case = inputs.stress(188, 8)
    B, Hkv, L, D = case.k_cache.shape
    ps = 16
    nb = L // ps
    g = torch.Generator().manual_seed(0)
    table = torch.randperm(B * nb, generator=g).view(B, nb).to(torch.int32)
    inv = torch.empty_like(table.view(-1))
    inv[table.view(-1).long()] = torch.arange(B * nb, dtype=torch.int32)
    pool_k = case.k_cache.view(B, Hkv, nb, ps, D).permute(0, 2, 1, 3, 4).reshape(B * nb, Hkv, ps, D)
    kp = pool_k[inv.long().cuda()].contiguous()
    del pool_k
    pool_v = case.v_cache.view(B, Hkv, nb, ps, D).permute(0, 2, 1, 3, 4).reshape(B * nb, Hkv, ps, D)
    vp = pool_v[inv.long().cuda()].contiguous()
    del pool_v
    out, lse = swa_verify_attn_paged(case.q, kp, vp, table.cuda(), case.seq_lens, case.q_pos,
                                     case.window, case.scale)
    torch.cuda.synchronize()
    del kp, vp
    seqs = _sample(case, 10, 52)
    ref_o, ref_l = oracle_reference(case, seqs)
    compare(out[seqs], lse[seqs], ref_o, ref_l, "paged stress_w188_q8, 16-row pages")
    del case
    torch.cuda.empty_cache()


def test_append_stress_full_size_sampled():
    from sliding_window_speculative_gb300 import swa_append_verify_attn
    case = inputs.stress(188, 8)
    B, q_len = case.q.shape[:2]
    Hkv, L, D = case.k_cache.shape[1:]
    seqs = _sample(case, 10, 53)
    ref_o, ref_l = oracle_reference(case, seqs)
    k_new = torch.empty((B, q_len, Hkv, D), dtype=torch.bfloat16, device="cuda")
    v_new = torch.empty_like(k_new)
    for b, qp in enumerate(case.q_pos_host):
        k_new[b] = case.k_cache[b, :, qp:qp + q_len].transpose(0, 1)
        v_new[b] = case.v_cache[b, :, qp:qp + q_len].transpose(0, 1)
        case.k_cache[b, :, qp:qp + q_len] = 1.0e4
        case.v_cache[b, :, qp:qp + q_len] = -1.0e4
    out, lse = swa_append_verify_attn(case.q, k_new, v_new, case.k_cache, case.v_cache,
                                      case.seq_lens, case.q_pos, case.window, case.scale)
    torch.cuda.synchronize()
    compare(out[seqs], lse[seqs], ref_o, ref_l, "fused append stress_w188_q8")
    for b in seqs:
        qp, sl = case.q_pos_host[b], case.seq_lens_host[b]
        lo = max(0, qp - 70)
        blk_k = case.k_cache[b, :, lo:sl].to(torch.float64).cpu().numpy()[None]
        blk_v = case.v_cache[b, :, lo:sl].to(torch.float64).cpu().numpy()[None]
        rows_k = k_new[b:b + 1].to(torch.float64).cpu().numpy()
        rows_v = v_new[b:b + 1].to(torch.float64).cpu().numpy()
        # the oracle's append on the slice before the call: poison rows
        # replaced by the block, everything else unchanged
        before_k = blk_k.copy()
        before_k[0, :, qp - lo:sl - lo] = 1.0e4
        before_v = blk_v.copy()
        before_v[0, :, qp - lo:sl - lo] = -1.0e4
        exp_k = oracle.append_rows(before_k, rows_k, [qp - lo], [sl - lo])
        exp_v = oracle.append_rows(before_v, rows_v, [qp - lo], [sl - lo])
        assert np.array_equal(blk_k, exp_k) and np.array_equal(blk_v, exp_v), b
    del case, k_new, v_new
    torch.cuda.empty_cache()


@pytest.mark.parametrize("window", [188, 512, 1024])
@pytest.mark.parametrize("q_len", [1, 8])
def test_stress_every_sequence(window, q_len):
    case = inputs.stress(window, q_len)
    out, lse = run_gpu(case)
    ref_o, ref_l = oracle_reference(case)
    compare(out, lse, ref_o, ref_l, f"stress_w{window}_q{q_len}, all sequences")
    del case, out, lse
    torch.cuda.empty_cache()


@pytest.mark.parametrize("window", [188, 512, 1024])
def test_stress_q64_sixty_four_sequences(window):
    case = inputs.stress(window, 64)
    out, lse = run_gpu(case)
    seqs = _sample(case, 62, 54 + window)
    ref_o, ref_l = oracle_reference(case, seqs)
    compare(out[seqs], lse[seqs], ref_o, ref_l, f"stress_w{window}_q64, {len(seqs)} sequences")
    del case, out, lse
    torch.cuda.empty_cache()
