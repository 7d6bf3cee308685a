"""Parity of each CUDA step against the oracle, through the C ABI's test hooks:
dequantisation and the activation quantiser bit for bit, router indices bit
for bit (near ties redrawn), the permutation bit for bit, and the LRU slot
table bit for bit."""
import numpy as np
import pytest
import torch

from helpers import bf16_tensor, need_gpu, oracle_layer, reject_near_ties, small_spec
from oracle import layer as npl
from oracle.native import formats, quant
from oracle.native import layer as olayer
from oracle.native.lru import SlotTable
from routed_expert_layer_gemv_gb300 import capi
from routed_expert_layer_gemv_gb300 import workloads as wl
from routed_expert_layer_gemv_gb300.layer import build_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    need_gpu()


# ---------------------------------------------------------------- formats

@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4", "mxfp8", "bf16"])
def test_dequant_slot_bit_exact(fmt):
    spec = small_spec(E=4, n_slots=3, d_model=384, d_ff=256, fmt=fmt, has_shared=True)
    L = build_layer(spec, 21, 8)
    L.install(2, 1)
    L.install(0, 2)
    torch.cuda.synchronize()
    for slot, e, shared in ((1, 2, False), (2, 0, False), (-1, 0, True)):
        w = wl.expert_weights(spec, 21, e, shared=shared)
        for m, name in enumerate(("gate", "up", "down")):
            mat = w[name]
            out = torch.empty(mat.rows, mat.K, dtype=torch.float32, device="cuda")
            capi.moe_debug_dequant(L.h, slot, m, out)
            ref = formats.dequant(mat.codes, mat.scales, mat.tscale, fmt)
            assert np.array_equal(out.cpu().numpy().astype(np.float64), ref), (slot, name)
    L.close()


def _quant_inputs(rows, K, seed):
    g = np.random.default_rng(seed)
    v = g.standard_normal((rows, K)) * np.exp(g.uniform(-8, 8, (rows, 1)))
    v[0, :40] = 0.0                           # zero block + partial
    v[1, :] = -1e-30                          # rounds to -0
    v[2, ::3] = 6.0 * 2.0 ** -3               # exact grid values
    v[3, :] = g.choice([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], K) * np.sign(g.standard_normal(K))
    v[4, :] *= 1e25
    return v.astype(np.float32)


@pytest.mark.parametrize("fmt,g_x", [("mxfp4", 1.0), ("nvfp4", 1.0), ("nvfp4", 0.25), ("mxfp8", 1.0), ("bf16", 1.0)])
def test_activation_quantiser_bit_exact(fmt, g_x):
    spec = small_spec(fmt=fmt)
    from routed_expert_layer_gemv_gb300.layer import MoELayer
    L = MoELayer(spec, 8, act_scale_x=g_x, act_scale_h=g_x)
    rows, K = 64, 512
    v = _quant_inputs(rows, K, 4)
    if fmt == "mxfp8":
        # E4M3 ties (1.0625, 1.1875), a value between grid points (248) and one
        # past the largest (464, saturating at 448); block exponent 0 for row 3
        g = np.random.default_rng(1)
        v[3, :] = g.choice([1.0625, 1.1875, 248.0, 464.0], K) * np.sign(g.standard_normal(K))
        v[5, :32] = 500.0
    blk = {"mxfp4": 32, "nvfp4": 16, "mxfp8": 32, "bf16": 32}[fmt]
    cbytes = {"mxfp4": K // 2, "nvfp4": K // 2, "mxfp8": K, "bf16": 2 * K}[fmt]
    vt = torch.from_numpy(v).cuda()
    codes = torch.empty(rows, cbytes, dtype=torch.uint8, device="cuda")
    scales = torch.empty(rows, K // blk, dtype=torch.uint8, device="cuda")
    capi.moe_debug_actquant(L.h, vt, rows, K, codes, scales, 0)
    if fmt == "bf16":
        # bf16 activations: the rounding of each value, nearest even
        got = codes.cpu().numpy().view("<u2").astype(np.uint32) << 16
        assert np.array_equal(got.view(np.float32).astype(np.float64), quant.round_bf16(v.astype(np.float64)))
        L.close()
        return
    if fmt == "mxfp4":
        rc, rs = quant.quant_mxfp4(v)
    elif fmt == "mxfp8":
        rc, rs = quant.quant_mxfp8(v)
    else:
        rc, rs = quant.quant_nvfp4(v, g_x)
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)
    L.close()


# ---------------------------------------------------------------- router

@pytest.mark.parametrize("case", [
    dict(spec=small_spec(router_std=1 / 16), N=64),
    dict(spec=wl.DECODE_35B.layer, N=40),
    dict(spec=wl.PREFILL_753B.layer, N=24),                         # bias, E=256, d=6144
    dict(spec=small_spec(E=32, k=6, d_model=512, norm_topk=False), N=33),
    dict(spec=small_spec(E=16, k=16, n_slots=16), N=5),             # k = E
    dict(spec=wl.DECODE_284B.layer, N=150),                          # tensor-core logits
    dict(spec=wl.PREFILL_753B.layer, N=200),                         # 2 expert tiles, ragged tokens
    dict(spec=small_spec(E=32, k=6, d_model=512, norm_topk=False), N=130),   # E below one tile
    dict(spec=wl.DECODE_35B.layer, N=65),                            # one token past the decode router
])
def test_router_indices_bit_exact(case):
    spec, N = case["spec"], case["N"]
    seed = 5
    W_r, b = wl.router_weights(spec, seed)
    from routed_expert_layer_gemv_gb300.layer import MoELayer
    L = MoELayer(spec, N)
    L.set_router(W_r, b)
    x, _ = wl.iid_tokens(seed, N, spec.d_model, reject_near_ties(spec, seed))
    xt = bf16_tensor(x)
    idx = torch.empty(N, spec.k, dtype=torch.int32, device="cuda")
    gates = torch.empty(N, spec.k, dtype=torch.float32, device="cuda")
    logits = torch.empty(N, spec.E, dtype=torch.float32, device="cuda")
    capi.moe_debug_router(L.h, xt, N, idx, gates, logits)
    ridx, rg, rL = olayer.router(wl.bf16_bits_to_f64(x), W_r, b, spec.k, spec.norm_topk)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.allclose(gates.cpu().numpy(), rg, rtol=2e-6, atol=1e-7)
    assert np.allclose(logits.cpu().numpy(), rL, rtol=1e-4, atol=2e-5)
    L.close()


@pytest.mark.parametrize("case", [
    dict(spec=small_spec(E=32, k=6, d_model=512), N=7),               # one entry per lane
    dict(spec=wl.DECODE_35B.layer, N=9),                              # decode router, E = 128
    dict(spec=wl.DECODE_35B.layer, N=130),                            # tensor-core logits, E = 128
    dict(spec=wl.PREFILL_753B.layer, N=40),                           # E = 256, bias
    dict(spec=small_spec(E=512, k=8, d_model=256, n_slots=64), N=20),  # E above 256, decode router
    dict(spec=small_spec(E=512, k=8, d_model=256, n_slots=64), N=70),  # E above 256, prefill top-k
])
def test_router_exact_ties_go_to_lower_id(case):
    """Exact ties: router rows (and biases) repeat in groups of G, so the
    logits of a group are equal bit for bit; G does not divide k, so a group
    straddles the k-th place.  The ids must be the k largest of the library's
    own logits with ties to the lower id (the oracle's selection run on them),
    and the gates their softmax."""
    spec, N = case["spec"], case["N"]
    G = 3 if spec.k % 3 else 4
    base = (np.arange(spec.E) // G) * G
    W_r, b = wl.router_weights(spec, 11)
    W_r = np.ascontiguousarray(W_r[base])
    if b is not None:
        b = np.ascontiguousarray(b[base])
    from routed_expert_layer_gemv_gb300.layer import MoELayer
    L = MoELayer(spec, N)
    L.set_router(W_r, b)
    x, _ = wl.iid_tokens(11, N, spec.d_model, None)
    idx = torch.empty(N, spec.k, dtype=torch.int32, device="cuda")
    gates = torch.empty(N, spec.k, dtype=torch.float32, device="cuda")
    logits = torch.empty(N, spec.E, dtype=torch.float32, device="cuda")
    capi.moe_debug_router(L.h, bf16_tensor(x), N, idx, gates, logits)
    Lg = logits.cpu().numpy().astype(np.float64)
    assert np.array_equal(Lg, Lg[:, base])                             # the ties are exact
    ridx = npl.topk_select(Lg, spec.k)
    got = idx.cpu().numpy()
    assert np.array_equal(got, ridx)
    # a group on the k-th place keeps its lower members
    straddles = 0
    for t in range(N):
        sel = set(got[t].tolist())
        assert all(e - 1 in sel for e in sel if e % G)
        straddles += any(e + 1 not in sel and (e + 1) % G and e + 1 < spec.E for e in sel)
    assert straddles >= N // 2
    m = Lg.max(axis=1, keepdims=True)
    p = np.exp(Lg - m)
    sel = np.take_along_axis(p, ridx, axis=1)
    rg = sel / sel.sum(axis=1, keepdims=True) if spec.norm_topk else sel / p.sum(axis=1, keepdims=True)
    assert np.allclose(gates.cpu().numpy(), rg, rtol=2e-6, atol=1e-7)
    L.close()


# ---------------------------------------------------------------- permute

@pytest.mark.parametrize("E,k,N", [(8, 2, 1), (8, 2, 64), (128, 8, 128), (128, 8, 129),
                                   (256, 8, 1000), (128, 8, 4096), (16, 16, 300), (1, 1, 7)])
def test_permute_bit_exact(E, k, N):
    g = np.random.default_rng(E * 7 + N)
    # skewed expert popularity, rows sorted ascending (as the router emits)
    p = g.dirichlet(np.ones(E) * 0.3)
    idx = np.stack([np.sort(g.choice(E, k, replace=False, p=p)) for _ in range(N)]).astype(np.int32)
    spec = small_spec(E=E, k=k, n_slots=E)
    from routed_expert_layer_gemv_gb300.layer import MoELayer
    L = MoELayer(spec, N)
    it = torch.from_numpy(idx).cuda()
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    row_of = torch.empty(N * k, dtype=torch.int32, device="cuda")
    tok_of = torch.empty(N * k, dtype=torch.int32, device="cuda")
    capi.moe_debug_permute(L.h, it, N, counts, offsets, row_of, tok_of)
    rc, ro, rr, rt = olayer.permute(idx, E)
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(row_of.cpu().numpy(), rr.reshape(-1))
    assert np.array_equal(tok_of.cpu().numpy(), rt)
    L.close()


# ---------------------------------------------------------------- LRU

def _state(L, S):
    eo, st, clk = capi.moe_lru_get_state(L.h, S)
    return eo, st, clk


@pytest.mark.parametrize("E,S,per_step,steps", [(8, 3, 2, 60), (128, 47, 8, 120), (128, 47, 70, 40),
                                                (256, 28, 20, 60), (16, 16, 9, 40)])
def test_lru_touch_matches_slot_table(E, S, per_step, steps):
    spec = small_spec(E=E, k=min(8, E), n_slots=S)
    from routed_expert_layer_gemv_gb300.layer import MoELayer
    L = MoELayer(spec, 64)
    T = SlotTable(E, S)
    g = np.random.default_rng(E + S)
    hot = g.choice(E, min(E, 2 * S), replace=False)
    for step in range(steps):
        pool = hot if g.random() < 0.7 else np.arange(E)
        routed = [int(v) for v in g.choice(pool, min(per_step, len(pool)), replace=False)]
        routed = routed + routed[:3]                      # duplicates count once
        slots, me, ms = capi.moe_lru_touch(L.h, routed)
        acc = T.step(routed)
        where = {e: s for e, s, _, _ in acc}
        assert slots == [where[e] for e in routed]
        assert me == [e for e, _, hit, _ in acc if not hit]
        assert ms == [s for _, s, hit, _ in acc if not hit]
        eo, st, clk = _state(L, S)
        assert eo == T.expert_of and st == T.stamp and clk == T.clock
    L.close()


@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4"])
def test_lru_touch_fills_land_in_their_slots(fmt):
    # touches of more distinct experts than slots (several waves) with a host
    # pool: every slot must then hold, bit for bit, the expert the table names
    spec = small_spec(E=20, k=4, d_model=256, d_ff=256, n_slots=5, fmt=fmt)
    seed = 17
    L = build_layer(spec, seed, 16)
    T = SlotTable(spec.E, spec.n_slots)
    g = np.random.default_rng(5)
    for step in range(6):
        routed = [int(v) for v in g.choice(spec.E, int(g.integers(3, 14)), replace=False)]
        capi.moe_lru_touch(L.h, routed)
        T.step(routed)
        eo, _, _ = _state(L, spec.n_slots)
        assert eo == T.expert_of
        for slot, e in enumerate(eo):
            if e < 0:
                continue
            w = wl.expert_weights(spec, seed, e)
            for m, name in enumerate(("gate", "up", "down")):
                mat = w[name]
                out = torch.empty(mat.rows, mat.K, dtype=torch.float32, device="cuda")
                capi.moe_debug_dequant(L.h, slot, m, out)
                ref = formats.dequant(mat.codes, mat.scales, mat.tscale, fmt)
                assert np.array_equal(out.cpu().numpy().astype(np.float64), ref), (step, slot, e, name)
    L.close()


def test_lru_install_and_state_roundtrip():
    spec = small_spec(E=10, k=2, n_slots=4)
    L = build_layer(spec, 1, 8)
    T = SlotTable(10, 4)
    for e, s in ((3, 0), (7, 1), (3, 2), (9, 1)):
        L.install(e, s)
        T.install(e, s)
    torch.cuda.synchronize()
    eo, st, clk = _state(L, 4)
    assert eo == T.expert_of and st == T.stamp and clk == T.clock
    capi.moe_lru_set_state(L.h, [5, -1, 2, 8], [4, 0, 9, 2], 11)
    eo, st, clk = _state(L, 4)
    assert eo == [5, -1, 2, 8] and st == [4, 0, 9, 2] and clk == 11
    with pytest.raises(capi.MoeError):
        capi.moe_lru_set_state(L.h, [5, 5, 2, 8], [4, 0, 9, 2], 11)   # expert twice
    with pytest.raises(capi.MoeError):
        L.install(10, 0)                                                # expert out of range
    L.close()


# ---------------------------------------------------------------- decode GEMV decode

@pytest.mark.parametrize("spec,N", [
    (small_spec(E=8, k=2, d_model=512, d_ff=256, n_slots=8, has_shared=True), 8),
    (small_spec(E=16, k=4, d_model=512, d_ff=384, n_slots=16, fmt="nvfp4", has_shared=True), 12),
    (small_spec(E=128, k=8, d_model=2048, d_ff=768, n_slots=128), 4),
    (small_spec(E=8, k=2, d_model=512, d_ff=384, n_slots=8, fmt="mxfp8", has_shared=True), 8),
    (small_spec(E=8, k=2, d_model=384, d_ff=256, n_slots=8, fmt="bf16", has_shared=True), 6),
])
def test_decode_gemv_decodes_weights_bit_exact(spec, N):
    # one-hot tokens x_t = c_t e_{i_t} (c_t a power of two): phase 1 of the
    # decode expert GEMV then writes, for each row of expert e and token t,
    # exactly c_t times column i_t of e's dequantised gate and up matrices --
    # the GEMV's own FP4 decode (E2M1 codes, block scales, tensor scale) is
    # checked bit for bit, not through the output tolerance
    seed = 41
    L = build_layer(spec, seed, N, install_all=True)
    g = np.random.default_rng(3)
    cols = g.choice(spec.d_model, N, replace=False)
    mags = [1.0, 0.125, 32.0, -2.0, -0.25, 4.0]
    xf = np.zeros((N, spec.d_model), dtype=np.float32)
    for t in range(N):
        xf[t, cols[t]] = mags[t % len(mags)]
    bits = (xf.view(np.uint32) >> 16).astype(np.uint16)          # exact in bf16
    L.forward(bf16_tensor(bits), regime=capi.MOE_REGIME_DECODE)
    rows = N * spec.k + (N if spec.has_shared else 0)
    hid = torch.empty(rows, 2 * spec.d_ff, dtype=torch.float32, device="cuda")
    capi.moe_debug_last_hidden(L.h, hid)
    idx = torch.empty(N * spec.k, dtype=torch.int32, device="cuda")
    row_of = torch.empty(N * spec.k, dtype=torch.int32, device="cuda")
    capi.moe_debug_last_step(L.h, idx=idx, row_of=row_of)
    torch.cuda.synchronize()
    H, I, R = hid.cpu().numpy().astype(np.float64), idx.cpu().numpy(), row_of.cpu().numpy()
    f = spec.d_ff
    cache = {}

    def deq(e, shared=False):
        key = (e, shared)
        if key not in cache:
            w = wl.expert_weights(spec, seed, e, shared=shared)
            cache[key] = {n: formats.dequant(m.codes, m.scales, m.tscale, spec.fmt) for n, m in w.items()}
        return cache[key]

    for t in range(N):
        c = float(xf[t, cols[t]])
        for j in range(spec.k):
            W = deq(int(I[t * spec.k + j]))
            r = R[t * spec.k + j]
            assert np.array_equal(H[r, :f], c * W["gate"][:, cols[t]]), (t, j, "gate")
            assert np.array_equal(H[r, f:], c * W["up"][:, cols[t]]), (t, j, "up")
        if spec.has_shared:
            W = deq(0, shared=True)
            r = N * spec.k + t
            assert np.array_equal(H[r, :f], c * W["gate"][:, cols[t]]), (t, "shared gate")
            assert np.array_equal(H[r, f:], c * W["up"][:, cols[t]]), (t, "shared up")
    L.close()
