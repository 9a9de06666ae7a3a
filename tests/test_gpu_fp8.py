"""GPU parity of the fp8 (E4M3) KV cache against the oracle.

Cache writes and block copies must match the oracle byte for byte (the
quantisation included); decode attention over the codes must meet the same
bar as the bf16 path, element by element against the fp64 oracle over the
same codes: |gpu - ref| <= 1e-2 and |gpu - ref| / max(|ref|, 1e-2) <= 2e-2,
and every (sequence, head) row within 2e-2 relative L2 error."""
import numpy as np
import pytest
import torch

from oracle import paref
from paged_kv_cache_105_gb300 import binding as B
from paged_kv_cache_105_gb300 import workloads as W
from tests.helpers import (bits, compare, gpu_step_fp8, oracle_step_fp8, sampled_oracle,
                           to_dev)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
KS, VS = W.FP8_SCALE, W.FP8_SCALE


def full_parity_fp8(wl, k_scale=KS, v_scale=VS, poison=True):
    vals_cpu = W.make_values_fp8(wl, poison_tails=poison, k_scale=k_scale, v_scale=v_scale)
    ref, kp, vp = oracle_step_fp8(wl, vals_cpu, k_scale, v_scale)
    vals = {k: v.to(DEV) for k, v in vals_cpu.items()}
    out, err = gpu_step_fp8(wl, vals, k_scale, v_scale)
    assert err == 0
    assert np.array_equal(vals["k_pool"].cpu().numpy(), kp)
    assert np.array_equal(vals["v_pool"].cpu().numpy(), vp)
    return compare(out, ref, wl.name + "-fp8")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_fp8_cache_write_bit_exact(d, bs):
    rng = np.random.default_rng(d + bs)
    T, Hkv, NB = 300, 4, 64
    g = torch.Generator().manual_seed(d * 100 + bs)
    k = torch.randn((T, Hkv, d), generator=g, dtype=torch.float32)
    v = torch.randn((T, Hkv, d), generator=g, dtype=torch.float32)
    # saturating, tiny (subnormal codes, signed zeros) and ordinary rows
    k[0:20] *= 50.0
    v[20:40] *= 1e-4
    k[40:60] *= 1e-6
    k, v = k.to(torch.bfloat16), v.to(torch.bfloat16)
    slots = rng.permutation(NB * bs)[:T].astype(np.int32)
    slots[5] = -1
    slots[7] = NB * bs + 3  # out of range: skipped and flagged
    k_scale, v_scale = np.float32(0.0123), np.float32(3.7e-3)
    kp0 = torch.randint(0, 256, (NB, Hkv, bs, d), generator=g, dtype=torch.uint8)
    vp0 = torch.randint(0, 256, (NB, Hkv, bs, d), generator=g, dtype=torch.uint8)
    kp_ref, vp_ref = kp0.numpy().copy(), vp0.numpy().copy()
    skipped = paref.reshape_and_cache_fp8(bits(k), bits(v), kp_ref, vp_ref, slots, k_scale,
                                          v_scale)
    assert skipped == 1
    kp, vp = kp0.to(DEV), vp0.to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.pa_reshape_and_cache_fp8(k.to(DEV), v.to(DEV), kp, vp, torch.from_numpy(slots).to(DEV),
                               float(k_scale), float(v_scale), err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == B.PA_DEV_ERR_SLOT
    assert np.array_equal(kp.cpu().numpy(), kp_ref)
    assert np.array_equal(vp.cpu().numpy(), vp_ref)
    # the saturating rows really saturated, the tiny ones produced signed zeros
    assert (kp_ref == 0x7E).any() and (kp_ref == 0xFE).any() and (kp_ref == 0x80).any()


def test_fp8_copy_blocks_bit_exact():
    g = torch.Generator().manual_seed(5)
    NB, Hkv, bs, d = 40, 2, 16, 128
    kp0 = torch.randint(0, 256, (NB, Hkv, bs, d), generator=g, dtype=torch.uint8)
    vp0 = torch.randint(0, 256, (NB, Hkv, bs, d), generator=g, dtype=torch.uint8)
    pairs = np.array([[3, 10], [11, 4], [0, 39], [7, 50]], np.int32)
    kr, vr = kp0.numpy().copy(), vp0.numpy().copy()
    assert paref.copy_blocks(kr.view(np.uint16), vr.view(np.uint16), pairs) == 1
    kp, vp = kp0.to(DEV), vp0.to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.pa_copy_blocks_fp8(kp, vp, torch.from_numpy(pairs).to(DEV), err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == B.PA_DEV_ERR_PAIR
    assert np.array_equal(kp.cpu().numpy(), kr) and np.array_equal(vp.cpu().numpy(), vr)


LENS = [1, 2, 15, 16, 17, 31, 33, 100, 257, 0, 1000, 2049, 64, 5]


@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("heads", [(8, 8), (32, 8), (16, 1), (12, 1)])
def test_fp8_decode_length_mix(bs, heads):
    Hq, Hkv = heads
    wl = W.custom(LENS, block_size=bs, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=128,
                  seed=bs * 7 + Hq, name=f"fp8-mix-bs{bs}-q{Hq}kv{Hkv}")
    full_parity_fp8(wl)


def test_fp8_gqa_batch_config():
    full_parity_fp8(W.config2())


def test_fp8_prefix_sharing_config():
    wl = W.config4()
    assert len(wl.cow_pairs) > 100
    full_parity_fp8(wl)


def test_fp8_scales_apply():
    # a power-of-two change of both scales scales nothing but the output by
    # the V factor (scores: the K factor is absorbed by the softmax scale)
    wl = W.custom([40, 300, 7], n_q_heads=16, n_kv_heads=4, seed=11, name="fp8-scales")
    full_parity_fp8(wl, k_scale=0.25 * KS, v_scale=8.0 * VS)


def test_fp8_fragmented_mha_full_size_every_output():
    wl = W.config3(block_size=16)
    vals = W.make_values_fp8(wl, device=DEV, poison_tails=True)
    seqs = list(range(wl.num_seqs))
    ref = sampled_oracle(wl, vals, seqs, fp8_scales=(KS, VS))
    out, err = gpu_step_fp8(wl, vals, KS, VS)
    assert err == 0
    compare(out[seqs], ref, wl.name + "-fp8")


def test_fp8_long_context_full_size_every_output():
    wl = W.config5()
    vals = W.make_values_fp8(wl, device=DEV, poison_tails=True)
    seqs = list(range(wl.num_seqs))  # all 16 sequences, every head
    ref = sampled_oracle(wl, vals, seqs, fp8_scales=(KS, VS))
    out, err = gpu_step_fp8(wl, vals, KS, VS)
    assert err == 0
    compare(out[seqs], ref, wl.name + "-fp8")


def test_fp8_bad_block_id_flagged():
    wl = W.custom([40, 70], n_q_heads=8, n_kv_heads=2, seed=3, name="fp8-badid")
    wl.block_tables[1, 2] = wl.num_blocks + 5
    vals = {k: v.to(DEV) for k, v in W.make_values_fp8(wl).items()}
    out, err = gpu_step_fp8(wl, vals, KS, VS, run_writes=False)
    assert err & B.PA_DEV_ERR_BLOCK_ID
    assert torch.isfinite(out[0].float()).all()


def test_fp8_unsupported_and_invalid_arguments():
    wl = W.custom([10], n_q_heads=4, n_kv_heads=4, head_dim=64, seed=1, name="fp8-d64")
    vals = {k: v.to(DEV) for k, v in W.make_values_fp8(wl).items()}
    t = to_dev(wl, DEV)
    ws = B.decode_workspace(1, 4, 4, 64, 16, wl.max_seq_len, 0, device=DEV)
    out = torch.zeros_like(vals["q"])
    with pytest.raises(B.PAError) as e:
        B.pa_decode_fp8(out, vals["q"], vals["k_pool"], vals["v_pool"], t["block_tables"],
                        t["seq_lens"], wl.scale, KS, VS, max_seq_len=wl.max_seq_len,
                        workspace=ws)
    assert e.value.status == B.PA_ERR_UNSUPPORTED
    with pytest.raises(B.PAError) as e:
        B.pa_reshape_and_cache_fp8(vals["k_new"], vals["v_new"], vals["k_pool"], vals["v_pool"],
                                   t["slot_mapping"], 0.0, VS)
    assert e.value.status == B.PA_ERR_INVALID_ARG


def test_fp8_rising_scores_move_the_running_max():
    # codes drawn from N(0, 1) * (1 + 0.1 i) / scale: scores grow along the
    # sequence, so the running maximum keeps moving by large steps
    wl = W.custom([900, 250, 33], n_q_heads=16, n_kv_heads=4, seed=22, name="fp8-rising")
    k_scale = 0.25
    vals_cpu = W.make_values_fp8(wl, k_scale=k_scale)
    g = torch.Generator().manual_seed(7)
    kp = torch.randn(vals_cpu["k_pool"].shape, generator=g)
    kn = vals_cpu["k_new"].float()
    bs = wl.block_size
    for s in range(wl.num_seqs):
        L = int(wl.seq_lens[s])
        for i in range(L - 1):
            kp[int(wl.block_tables[s, i // bs]), :, i % bs, :] *= 1.0 + 0.1 * i
        kn[s] *= 1.0 + 0.1 * (L - 1)
    vals_cpu["k_pool"] = (kp / k_scale).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    vals_cpu["k_new"] = kn.to(torch.bfloat16)
    ref, _, _ = oracle_step_fp8(wl, vals_cpu, k_scale, VS)
    vals = {k: v.to(DEV) for k, v in vals_cpu.items()}
    out, err = gpu_step_fp8(wl, vals, k_scale, VS)
    assert err == 0
    compare(out, ref, "fp8-rising")


def test_fp8_prepared_step_matches_the_oracle():
    wl = W.config4()
    vals_cpu = W.make_values_fp8(wl, poison_tails=True)
    ref, kp, vp = oracle_step_fp8(wl, vals_cpu, KS, VS)
    vals = {k: v.to(DEV) for k, v in vals_cpu.items()}
    t = to_dev(wl, DEV)
    ws = B.decode_workspace(wl.num_seqs, wl.n_q_heads, wl.n_kv_heads, wl.head_dim,
                            wl.block_size, wl.max_seq_len, 0, device=DEV)
    out = torch.full_like(vals["q"], float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    step = B.DecodeStep(out, vals["q"], vals["k_pool"], vals["v_pool"], t["block_tables"],
                        t["seq_lens"], wl.scale, max_seq_len=wl.max_seq_len, workspace=ws,
                        k_new=vals["k_new"], v_new=vals["v_new"],
                        slot_mapping=t["slot_mapping"], pairs=t["pairs"], err_word=err,
                        kv_scales=(KS, VS))
    step.enqueue()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(vals["k_pool"].cpu().numpy(), kp)
    assert np.array_equal(vals["v_pool"].cpu().numpy(), vp)
    compare(out, ref, wl.name + "-fp8-prepared")
