"""Whole-layer parity of moe_forward against the FP64 oracle: small shapes
spanning several row blocks and ragged expert groups, LRU misses with fills
and overflow waves, the shared expert, NVFP4 with a router bias, determinism,
token-permutation invariance, host buffers and the error paths."""
import numpy as np
import pytest
import torch

from helpers import (CachedExperts, assert_close_layer, bf16_tensor, need_gpu, oracle_layer,
                     reject_near_ties, small_spec)
from oracle import formats
from oracle import layer as olayer
from oracle.lru import SlotTable
from routed_expert_layer_gemv_gb300 import capi
from routed_expert_layer_gemv_gb300 import workloads as wl
from routed_expert_layer_gemv_gb300.layer import MoELayer, build_layer

pytestmark = pytest.mark.gpu
DEC = capi.MOE_REGIME_DECODE


@pytest.fixture(autouse=True)
def _gpu():
    need_gpu()


def _tokens(spec, seed, N):
    x, _ = wl.iid_tokens(seed, N, spec.d_model, reject_near_ties(spec, seed))
    return x


@pytest.mark.parametrize("spec,N", [
    (wl.TINY.layer, 64),
    (wl.TINY.layer, 1),
    (small_spec(E=8, k=2, d_model=256, d_ff=512, n_slots=8, has_shared=True), 13),
    (small_spec(E=32, k=4, d_model=512, d_ff=256, n_slots=32, fmt="nvfp4", has_shared=True,
                has_bias=True), 21),
    (small_spec(E=16, k=16, d_model=384, d_ff=384, n_slots=16), 3),   # k = E
    (small_spec(E=1, k=1, d_model=256, d_ff=128, n_slots=1), 9),      # E = 1: dense SwiGLU
    (small_spec(E=4, k=2, d_model=6144, d_ff=256, n_slots=4, fmt="nvfp4", has_shared=True,
                has_bias=True), 12),                                  # wide K, 2 token groups
    (small_spec(E=4, k=2, d_model=6144, d_ff=384, n_slots=4), 3),     # wide K, odd tile count
])
def test_forward_all_resident(spec, N):
    seed = 11
    L = build_layer(spec, seed, N, install_all=True)
    x = _tokens(spec, seed, N)
    y, info = L.forward(bf16_tensor(x), regime=DEC)
    torch.cuda.synchronize()
    assert info.host_synced == 0 and info.n_misses == 0
    ref, _, _ = oracle_layer(spec, seed).forward(wl.bf16_bits_to_f64(x), "decode")
    assert_close_layer(y, ref, "%s N=%d" % (spec, N))
    L.close()


def _decode_run(spec, seed, batch, steps, check_every=1, fill=capi.MOE_FILL_MEMCPY):
    N = batch
    experts = CachedExperts(spec, seed, cap=96)
    L = build_layer(spec, seed, N, experts_fn=experts)
    capi.moe_set_fill_mode(L.h, fill)
    O = oracle_layer(spec, seed, experts)
    T = SlotTable(spec.E, spec.n_slots)
    xs, _ = wl.ar1_tokens(seed, batch, steps, spec.d_model, 0.9, reject_near_ties(spec, seed))
    tot_miss = tot_u = waves = 0
    for t in range(steps):
        xt = bf16_tensor(xs[t])
        y, info = L.forward(xt, regime=DEC)
        ref, idx, _ = O.forward(wl.bf16_bits_to_f64(xs[t]), "decode")
        acc = T.step(idx.reshape(-1))
        n_miss = sum(1 for a in acc if not a[2])
        eff = fill
        if fill == capi.MOE_FILL_AUTO:   # the library's per-call choice
            eff = capi.MOE_FILL_FUSED if min(spec.E, N * spec.k) <= spec.n_slots else capi.MOE_FILL_KERNEL
        if eff in (capi.MOE_FILL_MEMCPY, capi.MOE_FILL_KERNEL):
            assert info.host_synced == 1
            assert info.n_distinct == len(acc)
            assert info.n_misses == n_miss
            assert info.fill_bytes == info.n_misses * L.expert_bytes
            waves = max(waves, info.n_waves)
        else:
            assert info.host_synced == 0
            waves = max(waves, (len(acc) + spec.n_slots - 1) // spec.n_slots)
        tot_miss += n_miss
        tot_u += len(acc)
        if t % check_every == 0 or t == steps - 1:
            assert_close_layer(y, ref, "step %d" % t)
            eo, st, clk = capi.moe_lru_get_state(L.h, spec.n_slots)
            assert eo == T.expert_of and st == T.stamp and clk == T.clock
    steps_d, u_d, hits_d, miss_d = capi.moe_stats(L.h)
    assert (steps_d, u_d, miss_d) == (steps, tot_u, tot_miss) and hits_d == tot_u - tot_miss
    L.close()
    return tot_miss, tot_u, waves


def test_decode_35b_shape_with_misses():
    # the decode layer shape, batch 4, cold cache of 47 slots: fills each step
    spec = wl.DECODE_35B.layer
    miss, u, waves = _decode_run(spec, 3, 4, 10)
    assert miss > 0 and miss < u


def test_decode_overflow_waves():
    # batch 16 routes to more distinct experts than the 47 slots hold
    spec = wl.DECODE_35B.layer
    miss, u, waves = _decode_run(spec, 4, 16, 3)
    assert waves >= 2


def test_decode_284b_shape_shared_and_waves():
    spec = wl.DECODE_284B.layer
    miss, u, waves = _decode_run(spec, 5, 8, 3)
    assert waves >= 2


@pytest.mark.parametrize("fill", [capi.MOE_FILL_DEVICE, capi.MOE_FILL_KERNEL, capi.MOE_FILL_FUSED,
                                  capi.MOE_FILL_AUTO])
@pytest.mark.parametrize("batch,steps", [(1, 8), (4, 6), (16, 3)])
def test_decode_copy_kernel_fill(batch, steps, fill):
    # misses pulled from the pinned pool by the GPU: DEVICE by a copy kernel
    # that reads the routing record on the GPU (no host wait), KERNEL by one on
    # reserved SMs (chunked at batch 16), FUSED by the expert FFN itself, which
    # writes them on to their slots (checked through the LRU state and later hits)
    spec = wl.DECODE_35B.layer
    miss, u, waves = _decode_run(spec, 7, batch, steps, fill=fill)
    assert miss > 0


@pytest.mark.parametrize("fill", [capi.MOE_FILL_KERNEL, capi.MOE_FILL_FUSED])
def test_decode_284b_shape_kernel_fill(fill):
    # shared expert, d_model 4096 MXFP4 experts, more distinct experts than slots
    spec = wl.DECODE_284B.layer
    miss, u, waves = _decode_run(spec, 5, 8, 3, fill=fill)
    assert waves >= 2


@pytest.mark.parametrize("fill", [capi.MOE_FILL_MEMCPY, capi.MOE_FILL_DEVICE, capi.MOE_FILL_KERNEL,
                                  capi.MOE_FILL_FUSED])
@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4"])
def test_staged_misses_land_in_their_lru_slots(fill, fmt):
    # more distinct experts per step than slots: misses past the first wave are
    # filled into spare buffers that then become their slots' buffers; every
    # LRU slot must then hold exactly the expert the slot table names
    spec = small_spec(E=32, k=4, d_model=256, d_ff=256, n_slots=6, fmt=fmt, has_shared=True)
    seed, batch = 13, 8
    experts = CachedExperts(spec, seed)
    L = build_layer(spec, seed, batch, experts_fn=experts)
    capi.moe_set_fill_mode(L.h, fill)
    O = oracle_layer(spec, seed, experts)
    T = SlotTable(spec.E, spec.n_slots)
    xs, _ = wl.ar1_tokens(seed, batch, 3, spec.d_model, 0.9, reject_near_ties(spec, seed))
    overflow = 0
    for t in range(3):
        y, info = L.forward(bf16_tensor(xs[t]), regime=DEC)
        ref, idx, _ = O.forward(wl.bf16_bits_to_f64(xs[t]), "decode")
        acc = T.step(idx.reshape(-1))
        overflow += len(acc) > spec.n_slots
        assert_close_layer(y, ref, "step %d" % t)
        eo, _, _ = capi.moe_lru_get_state(L.h, spec.n_slots)
        assert eo == T.expert_of
        torch.cuda.synchronize()
        for slot, e in enumerate(eo):
            if e < 0:
                continue
            w = experts(e)
            for m, name in enumerate(("gate", "up", "down")):
                mat = w[name]
                out = torch.empty(mat.rows, mat.K, dtype=torch.float32, device="cuda")
                capi.moe_debug_dequant(L.h, slot, m, out)
                want = formats.dequant(mat.codes, mat.scales, mat.tscale, spec.fmt)
                assert np.array_equal(out.cpu().numpy().astype(np.float64), want), (t, slot, e, name)
    assert overflow > 0
    L.close()


@pytest.mark.parametrize("fill", [capi.MOE_FILL_DEVICE, capi.MOE_FILL_KERNEL, capi.MOE_FILL_FUSED])
def test_prefill_copy_kernel_fill_waves(fill):
    # KERNEL mode fills prefill misses with the copy engine (the GEMM holds every SM)
    spec = small_spec(E=24, k=3, d_model=512, d_ff=256, n_slots=5, fmt="nvfp4", has_shared=True,
                      has_bias=True)
    seed, N = 31, 96
    experts = CachedExperts(spec, seed)
    L = build_layer(spec, seed, N, experts_fn=experts)
    capi.moe_set_fill_mode(L.h, fill)
    O = oracle_layer(spec, seed, experts)
    for step in range(2):
        x = _tokens(spec, seed + step, N)
        y, info = L.forward(bf16_tensor(x), regime=capi.MOE_REGIME_PREFILL)
        assert info.host_synced == (0 if fill == capi.MOE_FILL_DEVICE else 1)
        ref, _, _ = O.forward(wl.bf16_bits_to_f64(x), "prefill")
        assert_close_layer(y, ref, "prefill device fill step %d" % step)
    L.close()


@pytest.mark.parametrize("fill", [capi.MOE_FILL_MEMCPY, capi.MOE_FILL_KERNEL, capi.MOE_FILL_FUSED])
def test_decode_nvfp4_bias_small_cache(fill):
    # d_ff 384: the down rows end in a half-filled 256-K box; later steps hit
    # the experts earlier misses left in the slots (tensor scales included)
    spec = small_spec(E=24, k=3, d_model=512, d_ff=384, n_slots=5, fmt="nvfp4", has_shared=True,
                      has_bias=True)
    miss, u, waves = _decode_run(spec, 6, 3, 12, fill=fill)
    assert miss > 0


def test_deterministic_bitwise():
    spec = wl.DECODE_35B.layer
    x = _tokens(spec, 8, 16)
    outs = []
    for _ in range(2):
        L = build_layer(spec, 8, 16)
        for e in range(40):
            L.install(e, e)
        y1, _ = L.forward(bf16_tensor(x), regime=DEC)
        y2, _ = L.forward(bf16_tensor(x), regime=DEC)
        torch.cuda.synchronize()
        outs += [y1.cpu(), y2.cpu()]
        L.close()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


def test_token_permutation_invariance_bitwise():
    spec = small_spec(E=16, k=4, d_model=512, d_ff=256, n_slots=16, has_shared=True)
    L = build_layer(spec, 9, 32, install_all=True)
    x = _tokens(spec, 9, 32)
    perm = np.random.default_rng(1).permutation(32)
    y, _ = L.forward(bf16_tensor(x), regime=DEC)
    yp, _ = L.forward(bf16_tensor(x[perm]), regime=DEC)
    torch.cuda.synchronize()
    assert torch.equal(yp.cpu().view(torch.int16), y.cpu()[perm].view(torch.int16))
    L.close()


def test_host_buffers_and_empty_batch():
    spec = wl.TINY.layer
    L = build_layer(spec, 12, 64, install_all=True)
    x = _tokens(spec, 12, 20)
    y_dev, _ = L.forward(bf16_tensor(x), regime=DEC)
    xh = bf16_tensor(x, device=None).pin_memory()
    yh = torch.empty(20, spec.d_model, dtype=torch.bfloat16).pin_memory()
    capi.moe_forward(L.h, xh, 20, yh, None, DEC)
    assert torch.equal(yh.view(torch.int16), y_dev.cpu().view(torch.int16))
    yp = torch.empty(20, spec.d_model, dtype=torch.bfloat16)          # pageable
    capi.moe_forward(L.h, xh, 20, yp, None, DEC)
    assert torch.equal(yp.view(torch.int16), y_dev.cpu().view(torch.int16))
    xp = bf16_tensor(x, device=None)                                   # pageable x: staged copy
    capi.moe_forward(L.h, xp, 20, yh, None, DEC)
    assert torch.equal(yh.view(torch.int16), y_dev.cpu().view(torch.int16))
    info = capi.moe_forward(L.h, xh, 0, yh, None, DEC)                # N = 0: no-op
    assert info.n_tokens == 0
    L.close()


def test_error_paths():
    spec = wl.TINY.layer
    L = MoELayer(spec, 8)
    x = torch.zeros(8, spec.d_model, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    with pytest.raises(capi.MoeError) as e:
        capi.moe_forward(L.h, x, 8, y, None, DEC)                      # router not set
    assert e.value.status == capi.MOE_ERR_STATE
    W_r, b = wl.router_weights(spec, 0)
    L.set_router(W_r, b)
    with pytest.raises(capi.MoeError) as e:
        capi.moe_forward(L.h, x, 8, y, None, DEC)                      # no pool, cache empty
    assert e.value.status == capi.MOE_ERR_NOT_INSTALLED
    with pytest.raises(capi.MoeError) as e:
        capi.moe_forward(L.h, x, 9, y, None, DEC)                      # N > max_tokens
    assert e.value.status == capi.MOE_ERR_ARG
    with pytest.raises(capi.MoeError) as e:
        capi.moe_forward(L.h, x, -1, y, None, DEC)
    assert e.value.status == capi.MOE_ERR_ARG
    with pytest.raises(capi.MoeError) as e:
        L.install(0, 0)                                                # no host pool
    assert e.value.status == capi.MOE_ERR_NOT_INSTALLED
    with pytest.raises(capi.MoeError) as e:
        capi.moe_set_shared_expert(L.h, x.data_ptr())                  # no shared expert
    assert e.value.status == capi.MOE_ERR_STATE
    L.close()


# ---------------------------------------------------------------- prefill regime

PRE = capi.MOE_REGIME_PREFILL


@pytest.mark.parametrize("spec,N", [
    (wl.TINY.layer, 64),
    (small_spec(E=16, k=4, d_model=512, d_ff=256, n_slots=16), 300),        # several ragged tiles
    (small_spec(E=32, k=4, d_model=512, d_ff=512, n_slots=32, fmt="nvfp4", has_shared=True,
                has_bias=True), 200),
    (small_spec(E=8, k=8, d_model=256, d_ff=256, n_slots=8), 130),           # k = E
])
def test_prefill_all_resident(spec, N):
    seed = 17
    L = build_layer(spec, seed, N, install_all=True)
    x = _tokens(spec, seed, N)
    y, info = L.forward(bf16_tensor(x), regime=PRE)
    torch.cuda.synchronize()
    assert info.regime == PRE
    ref, _, _ = oracle_layer(spec, seed).forward(wl.bf16_bits_to_f64(x), "prefill")
    assert_close_layer(y, ref, "prefill %s N=%d" % (spec, N))
    L.close()


def test_prefill_35b_shape_sampled_tokens():
    # the prefill layer shape (d 2048, E 128, top-8, d_ff 768) on 512 tokens
    spec = wl.PREFILL_35B.layer
    N, seed = 512, 19
    L = build_layer(spec, seed, N, install_all=True)
    x = _tokens(spec, seed, N)
    y, _ = L.forward(bf16_tensor(x), regime=PRE)
    torch.cuda.synchronize()
    sample = list(range(0, N, 37)) + [N - 1]
    ref, _, _ = oracle_layer(spec, seed).forward(wl.bf16_bits_to_f64(x), "prefill", tokens=sample)
    assert_close_layer(y[sample], ref, "prefill 35B shape")
    L.close()


def _full_chunk_parity(work, n_sample):
    # the bench's own prefill chunk (same generator, size and launch path),
    # checked on sampled tokens the oracle computes one expert at a time;
    # tokens whose k-th and (k+1)-th FP64 logits are within 1e-4 are skipped
    # (their expert choice is not unique at that tolerance)
    spec, N, seed = work.layer, work.n_tokens, work.seed
    x, _ = wl.iid_tokens(seed, N, spec.d_model)
    L = build_layer(spec, seed, N, install_all=True)
    y, info = L.forward(bf16_tensor(x), regime=PRE)
    torch.cuda.synchronize()
    assert info.regime == PRE
    W_r, b = wl.router_weights(spec, seed)
    cand = np.unique(np.linspace(0, N - 1, 4 * n_sample).astype(np.int64))
    tie = olayer.near_tie(wl.bf16_bits_to_f64(x[cand]), W_r, b, spec.k, 1e-4)
    sample = [int(t) for t, bad in zip(cand, tie) if not bad][:n_sample]
    assert len(sample) == n_sample
    ref, _, _ = oracle_layer(spec, seed).forward(wl.bf16_bits_to_f64(x[sample]), "prefill")
    assert_close_layer(y[sample], ref, "%s, sampled tokens" % work.name)
    L.close()


def test_prefill_35b_full_chunk_sampled():
    _full_chunk_parity(wl.PREFILL_35B, 12)


def test_prefill_753b_full_chunk_sampled():
    _full_chunk_parity(wl.PREFILL_753B, 4)


def test_prefill_with_misses_and_waves():
    spec = small_spec(E=24, k=3, d_model=512, d_ff=256, n_slots=5, fmt="nvfp4", has_shared=True,
                      has_bias=True)
    seed, N = 23, 96
    experts = CachedExperts(spec, seed)
    L = build_layer(spec, seed, N, experts_fn=experts)
    O = oracle_layer(spec, seed, experts)
    for step in range(3):
        x = _tokens(spec, seed + step, N)
        y, info = L.forward(bf16_tensor(x), regime=PRE)
        assert info.n_waves >= 2 and info.n_misses > 0
        ref, _, _ = O.forward(wl.bf16_bits_to_f64(x), "prefill")
        assert_close_layer(y, ref, "prefill waves step %d" % step)
    L.close()


def test_prefill_deterministic_bitwise():
    spec = small_spec(E=16, k=4, d_model=512, d_ff=256, n_slots=16, has_shared=True)
    x = _tokens(spec, 29, 200)
    outs = []
    for _ in range(2):
        L = build_layer(spec, 29, 200, install_all=True)
        y, _ = L.forward(bf16_tensor(x), regime=PRE)
        torch.cuda.synchronize()
        outs.append(y.cpu())
        L.close()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_auto_regime_picks_prefill_for_large_batches():
    spec = wl.TINY.layer
    L = build_layer(spec, 3, 128, install_all=True)
    x = _tokens(spec, 3, 128)
    _, info = L.forward(bf16_tensor(x))
    assert info.regime == PRE
    _, info = L.forward(bf16_tensor(x[:16]))
    assert info.regime == DEC
    L.close()
