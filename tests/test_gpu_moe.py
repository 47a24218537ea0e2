"""GPU parity of the mixture-of-experts path (w4a16_moe_align, w4a16_moe_linear,
w4a16_moe_sum) against the oracle: the alignment bit-exact, each slot's
expert linear within the linear's rule, the weighted sum within a bound
derived from its two roundings, and a whole expert MLP (gate+up with
SiLU-and-mul, down, sum) checked step by step on the GPU's own intermediates.

Routing is seeded: top-k distinct experts per token from a counter-based
permutation, weights a softmax of seeded logits over the chosen experts.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from helpers import assert_close

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def w4():
    import __graft_entry__
    __graft_entry__.build()
    import weight_only_int4_w4a16_gb300 as w4
    w4.w4a16_init(0, 512 << 20)
    return w4


@pytest.fixture(autouse=True)
def no_device_errors(request):
    yield
    if "w4" in request.fixturenames:
        import weight_only_int4_w4a16_gb300 as w4
        assert w4.w4a16_device_status() == 0, "a kernel reported an expired bounded wait"


def routing(seed, T, k, E):
    """ids [T, k] (distinct experts per token) and fp32 weights [T, k]."""
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    logits = rng.standard_normal((T, k))
    w = np.exp(logits - logits.max(axis=1, keepdims=True))
    w = (w / w.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids, w


def experts(seed, E, N, K, dev=DEV):
    """E seeded W4A16 layers stacked: qweight [E, N, K/8], scales [E, N, G], zeros."""
    parts = [si.layer(si.config_seed(seed, e), N, K, device=dev) for e in range(E)]
    return tuple(torch.stack([p[i] for p in parts]) for i in range(3))


def host(t):
    return t.detach().cpu().numpy()


def bits16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("T,k,E", [(1, 8, 128), (4, 8, 64), (64, 8, 128), (7, 3, 5), (32, 2, 4),
                                   (300, 8, 256)])
def test_align_matches_oracle(w4, T, k, E):
    ids, _ = routing(T * 1000 + k * 10 + E, T, k, E)
    srt, pos, off = w4.w4a16_moe_align(torch.from_numpy(ids).to(DEV), E)
    torch.cuda.synchronize()
    r_srt, r_pos, r_off = oracle.moe_align(ids, E)
    assert np.array_equal(host(off), r_off)
    assert np.array_equal(host(srt), r_srt)
    assert np.array_equal(host(pos), r_pos)


def test_align_flags_invalid_ids(w4):
    ids = np.array([[0, 3], [5, 1]], dtype=np.int32)  # 5 is not an expert of 4
    srt, pos, off = w4.w4a16_moe_align(torch.from_numpy(ids).to(DEV), 4)
    code = w4.w4a16_device_status()
    assert code & 1024
    assert host(off).tolist() == [0, 1, 2, 2, 3]
    assert host(pos)[2] == -1
    assert host(srt)[:3].tolist() == [0, 3, 1]


def run_moe_linear(w4, seed, T, k, E, N, K, epi=0, dt=torch.float16, per_slot=False):
    """One expert linear through the GPU path, and the oracle's (rows in sorted order)."""
    ids, _ = routing(seed, T, k, E)
    qw, s, zw = experts(seed, E, N, K)
    if dt == torch.bfloat16:
        s = s.float().to(dt)
    rows = T * k if per_slot else T
    x = si.x(si.config_seed(seed, 99), rows, K).float().to(dt)
    ex = w4.MoeExperts(qw, s, zw, epilogue=epi, max_slots=T * k)
    try:
        srt, pos, off = w4.w4a16_moe_align(torch.from_numpy(ids).to(DEV), E)
        xd = x.to(DEV)
        if per_slot:  # an input already in sorted order: row p is slot srt[p]'s
            xd = xd[srt.long()].contiguous()
        y = ex.linear(xd, srt, off, T * k, gather_k=0 if per_slot else k)
        torch.cuda.synchronize()
    finally:
        ex.destroy()
    name = "bf16" if dt == torch.bfloat16 else "f16"
    ref = oracle.moe_linear(bits16(x), host(qw).view(np.uint32), bits16(s), host(zw).view(np.uint32),
                            ids, per_slot=per_slot, dtype=name)
    if epi == w4.EPILOGUE_SILU_MUL:
        ref = oracle.silu_mul(ref)
    return y, ref[host(srt)], (ids, srt, pos, off)


# (T, k, E, N, K): decode with one token and 8 of 128 experts (a Qwen3-MoE-like
# expert MLP: hidden 2048, intermediate 768), several tokens, experts with more
# than 8 slots (several tiles), a split-K expert shape, ragged N
CASES = [(1, 8, 128, 768, 2048), (4, 8, 64, 1024, 2048), (32, 2, 4, 512, 1024),
         (3, 4, 16, 2048, 6144), (5, 2, 8, 777, 1408)]


@pytest.mark.parametrize("T,k,E,N,K", CASES)
def test_moe_linear_matches_oracle(w4, T, k, E, N, K):
    y, ref, _ = run_moe_linear(w4, T * 7 + E, T, k, E, N, K)
    assert_close(y, ref, f"moe T={T} k={k} E={E} N={N} K={K}")


@pytest.mark.parametrize("T,k,E,N,K", [(1, 8, 128, 1536, 2048), (16, 4, 8, 2048, 1024)])
def test_moe_gate_up_silu(w4, T, k, E, N, K):
    y, ref, _ = run_moe_linear(w4, T * 11 + E, T, k, E, N, K, epi=w4.EPILOGUE_SILU_MUL)
    assert_close(y, ref, f"moe silu T={T} E={E}")


def test_moe_input_in_sorted_order(w4):
    y, ref, _ = run_moe_linear(w4, 77, 4, 8, 32, 2048, 768, per_slot=True)
    assert_close(y, ref, "moe per-slot input")


def test_moe_bf16(w4):
    y, ref, _ = run_moe_linear(w4, 78, 4, 8, 32, 1024, 2048, dt=torch.bfloat16)
    assert_close(y, ref, "moe bf16")


def sum_tolerance(y_ref_slots, w, out_ref):
    """|out - out_ref| <= 1e-3 * max|out_ref| + 1e-3 (the linear's rule) plus
    what the per-slot outputs' own fp16 rounding and error can move the sum:
    their rule's bound weighted by |w|, elementwise."""
    T, k = w.shape
    tol_y = 1e-3 * np.abs(y_ref_slots).max() + 1e-3
    return 1e-3 * np.abs(out_ref).max() + 1e-3 + np.abs(w).sum(axis=1, keepdims=True) * tol_y


def test_moe_sum_matches_oracle(w4):
    T, k, N = 6, 4, 1000
    rng = np.random.default_rng(3)
    ys = torch.from_numpy(rng.standard_normal((T * k, N)) * 4).to(torch.float16)
    _, w = routing(4, T, k, 16)
    perm = rng.permutation(T * k).astype(np.int32)  # pos: slot -> row of ys
    out = w4.w4a16_moe_sum(ys.to(DEV), torch.from_numpy(perm).to(DEV), torch.from_numpy(w).to(DEV))
    torch.cuda.synchronize()
    y_slots = ys.double().numpy()[perm]
    ref = oracle.moe_sum(y_slots, w.astype(np.float64))
    err = np.abs(out.double().cpu().numpy() - ref)
    assert np.all(err <= sum_tolerance(y_slots, w, ref))


@pytest.mark.parametrize("T", [1, 4])
def test_moe_expert_mlp_step_by_step(w4, T):
    # x -> align -> gate+up (SiLU-and-mul, gathered by token) -> down (in
    # sorted order) -> weighted sum; each step against the oracle on the GPU's
    # own input to that step
    E, k, H, I = 32, 8, 1024, 768
    ids, w = routing(500 + T, T, k, E)
    g_qw, g_s, g_zw = experts(600, E, 2 * I, H)
    d_qw, d_s, d_zw = experts(601, E, H, I)
    x = si.x(si.config_seed(602, T), T, H)
    gate_up = w4.MoeExperts(g_qw, g_s, g_zw, epilogue=w4.EPILOGUE_SILU_MUL, max_slots=T * k)
    down = w4.MoeExperts(d_qw, d_s, d_zw, max_slots=T * k)
    try:
        srt, pos, off = w4.w4a16_moe_align(torch.from_numpy(ids).to(DEV), E)
        h = gate_up.linear(x.to(DEV), srt, off, T * k, gather_k=k)
        o = down.linear(h, srt, off, T * k, gather_k=0)
        out = w4.w4a16_moe_sum(o, pos, torch.from_numpy(w).to(DEV))
        torch.cuda.synchronize()
    finally:
        gate_up.destroy()
        down.destroy()
    order, slot_pos = host(srt), host(pos)
    h_ref = oracle.silu_mul(oracle.moe_linear(si.as_u16(x), host(g_qw).view(np.uint32),
                                              si.as_u16(g_s), host(g_zw).view(np.uint32), ids))
    assert_close(h, h_ref[order], "expert gate+up")
    h_slots = bits16(h)[slot_pos]  # the GPU's h, back in slot order
    o_ref = oracle.moe_linear(h_slots, host(d_qw).view(np.uint32), si.as_u16(d_s),
                              host(d_zw).view(np.uint32), ids, per_slot=True)
    assert_close(o, o_ref[order], "expert down")
    o_slots = o.double().cpu().numpy()[slot_pos]
    assert_close(out, oracle.moe_sum(o_slots, w.astype(np.float64)), "weighted sum")


@pytest.mark.parametrize("T,E,dt", [(1, 32, torch.float16), (4, 32, torch.float16),
                                    (8, 128, torch.float16), (4, 16, torch.bfloat16)])
def test_moe_mlp_one_launch_matches_the_chain(w4, T, E, dt):
    # w4a16_moe_mlp on its chain path (both linears in one expert-MMA launch,
    # down tiles waiting for their gate+up tiles) against the call-by-call
    # chain, which the test above checks against the oracle step by step, and
    # its intermediates against the oracle; run twice (the completion
    # counters must be left zeroed), bit-identical
    k, H, I = 8, 1024, 768
    ids, w = routing(800 + T + E, T, k, E)
    g_qw, g_s, g_zw = experts(610, E, 2 * I, H)
    d_qw, d_s, d_zw = experts(611, E, H, I)
    if dt == torch.bfloat16:
        g_s, d_s = g_s.float().to(dt), d_s.float().to(dt)
    x = si.x(si.config_seed(612, T), T, H).float().to(dt).to(DEV)
    ids_d, w_d = torch.from_numpy(ids).to(DEV), torch.from_numpy(w).to(DEV)
    gate_up = w4.MoeExperts(g_qw, g_s, g_zw, epilogue=w4.EPILOGUE_SILU_MUL, max_slots=T * k)
    down = w4.MoeExperts(d_qw, d_s, d_zw, max_slots=T * k)
    mlp = w4.MoeMlp(gate_up, down, T, k, path=w4.MOE_PATH_CHAIN)
    try:
        assert mlp.path(T) == w4.MOE_PATH_CHAIN
        outs = [mlp(x, ids_d, w_d) for _ in range(2)]
        torch.cuda.synchronize()
        h_m, o_m = (t.clone() for t in mlp.intermediates(T * k))
        srt, pos, off = w4.w4a16_moe_align(ids_d, E)
        h = gate_up.linear(x, srt, off, T * k, gather_k=k)
        o = down.linear(h, srt, off, T * k, gather_k=0)
        chain = w4.w4a16_moe_sum(o, pos, w_d)
        torch.cuda.synchronize()
    finally:
        mlp.destroy()
        gate_up.destroy()
        down.destroy()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert_close(outs[0], chain.double().cpu().numpy(), f"expert MLP T={T} E={E}")
    check_mlp_steps((g_qw, g_s, g_zw), (d_qw, d_s, d_zw), x.cpu(), ids, w, outs[0], h_m, o_m, E,
                    f"chain path T={T} E={E}")


# ---- the one-launch decode path of w4a16_moe_mlp ---------------------------

def mlp_experts(seed, E, H, I, dt):
    g = experts(seed, E, 2 * I, H)
    d = experts(seed + 1, E, H, I)
    if dt == torch.bfloat16:
        g = (g[0], g[1].float().to(dt), g[2])
        d = (d[0], d[1].float().to(dt), d[2])
    return g, d


def run_mlp(w4, g, d, x, ids, w, path):
    """One w4a16_moe_mlp call on a fresh handle: out, the path it took, and
    copies of its intermediate rows and expert outputs (sorted order)."""
    T, k = ids.shape
    gate_up = w4.MoeExperts(*g, epilogue=w4.EPILOGUE_SILU_MUL, max_slots=T * k)
    down = w4.MoeExperts(*d, max_slots=T * k)
    mlp = w4.MoeMlp(gate_up, down, T, k, path=path)
    try:
        taken = mlp.path(T)
        out = mlp(x.to(DEV), torch.from_numpy(ids).to(DEV), torch.from_numpy(w).to(DEV))
        torch.cuda.synchronize()
        h, o = (t.clone() for t in mlp.intermediates(T * k))
        torch.cuda.synchronize()
    finally:
        mlp.destroy()
        gate_up.destroy()
        down.destroy()
    return out, taken, h, o


def check_mlp_steps(g, d, x, ids, w, out, h, o, E, what):
    # each step against the oracle on the GPU's own input to that step:
    # h = silu(gate) * up in sorted order, o = down(h), out = the weighted sum
    r_srt, r_pos, _ = oracle.moe_align(ids, E)
    h_ref = oracle.silu_mul(oracle.moe_linear(bits16(x), host(g[0]).view(np.uint32), bits16(g[1]),
                                              host(g[2]).view(np.uint32), ids,
                                              dtype=name_of(x.dtype)))
    assert_close(h, h_ref[r_srt], f"{what}: gate+up")
    h_slots = bits16(h)[r_pos]
    o_ref = oracle.moe_linear(h_slots, host(d[0]).view(np.uint32), bits16(d[1]),
                              host(d[2]).view(np.uint32), ids, per_slot=True,
                              dtype=name_of(x.dtype))
    assert_close(o, o_ref[r_srt], f"{what}: down")
    o_slots = o.double().cpu().numpy()[r_pos]
    assert_close(out, oracle.moe_sum(o_slots, w.astype(np.float64)), f"{what}: weighted sum")


def name_of(dt):
    return "bf16" if dt == torch.bfloat16 else "f16"


# (T, k, E, H, I, dtype): a Qwen3-MoE-like decode expert MLP (hidden 2048,
# intermediate 768, top 8 of 128) at 1, 4 and 8 tokens; experts with several
# slots; bf16; a partial last stage in both linears (H 1152: 9 groups, two
# zeros words; I 384: 3 groups)
DECODE_CASES = [(1, 8, 128, 2048, 768, torch.float16), (4, 8, 128, 2048, 768, torch.float16),
                (8, 8, 64, 2048, 768, torch.float16), (2, 8, 16, 1024, 768, torch.bfloat16),
                (8, 8, 128, 2048, 768, torch.bfloat16), (3, 2, 8, 1152, 384, torch.float16)]


@pytest.mark.parametrize("T,k,E,H,I,dt", DECODE_CASES)
def test_moe_mlp_decode_matches_oracle(w4, T, k, E, H, I, dt):
    seed = 900 + 7 * T + E + I
    ids, w = routing(seed, T, k, E)
    g, d = mlp_experts(seed + 1, E, H, I, dt)
    x = si.x(si.config_seed(seed, 5), T, H).float().to(dt)
    out, taken, h, o = run_mlp(w4, g, d, x, ids, w, w4.MOE_PATH_AUTO)
    assert taken == w4.MOE_PATH_DECODE
    check_mlp_steps(g, d, x, ids, w, out, h, o, E, f"decode T={T} E={E} {name_of(dt)}")


def test_moe_mlp_decode_experts_with_many_slots(w4):
    # every token picks both experts twice: each expert has 16 slots (two
    # tiles of 8), and a tile holds two slots of one token
    T, k, E, H, I = 8, 4, 2, 1024, 512
    ids = np.tile(np.array([[0, 1, 0, 1]], dtype=np.int32), (T, 1))
    w = np.full((T, k), 0.25, dtype=np.float32)
    g, d = mlp_experts(950, E, H, I, torch.float16)
    x = si.x(si.config_seed(951), T, H)
    out, taken, h, o = run_mlp(w4, g, d, x, ids, w, w4.MOE_PATH_DECODE)
    assert taken == w4.MOE_PATH_DECODE
    check_mlp_steps(g, d, x, ids, w, out, h, o, E, "decode, 16 slots per expert")


def test_moe_mlp_decode_matches_chain_and_repeats(w4):
    # the decode path against the chain (each checked against the oracle
    # above), and three decode calls on one handle bit-identical (its
    # counters are left zeroed)
    T, k, E, H, I = 4, 8, 64, 2048, 768
    ids, w = routing(960, T, k, E)
    g, d = mlp_experts(961, E, H, I, torch.float16)
    x = si.x(si.config_seed(962), T, H).to(DEV)
    ids_d, w_d = torch.from_numpy(ids).to(DEV), torch.from_numpy(w).to(DEV)
    gate_up = w4.MoeExperts(*g, epilogue=w4.EPILOGUE_SILU_MUL, max_slots=T * k)
    down = w4.MoeExperts(*d, max_slots=T * k)
    mlp = w4.MoeMlp(gate_up, down, T, k)
    try:
        outs = [mlp(x, ids_d, w_d) for _ in range(3)]
        mlp.set_path(w4.MOE_PATH_CHAIN)
        chain = mlp(x, ids_d, w_d)
        torch.cuda.synchronize()
    finally:
        mlp.destroy()
        gate_up.destroy()
        down.destroy()
    for y in outs[1:]:
        assert torch.equal(y.view(torch.int16), outs[0].view(torch.int16))
    assert_close(outs[0], chain.double().cpu().numpy(), "decode vs chain")


def test_moe_mlp_decode_invalid_id_is_left_out(w4):
    # a slot whose id is not an expert sets the status bit and drops out of
    # the sum: out equals the call with that slot on expert 0 at weight 0
    # (an MMA column does not depend on the tile's other columns)
    T, k, E, H, I = 2, 4, 8, 1024, 512
    ids, w = routing(970, T, k, E)
    g, d = mlp_experts(971, E, H, I, torch.float16)
    x = si.x(si.config_seed(972), T, H)
    bad = ids.copy()
    bad[1, 2] = E
    out_bad, _, _, _ = run_mlp(w4, g, d, x, bad, w, w4.MOE_PATH_DECODE)
    code = w4.w4a16_device_status()
    assert code & 1024
    fixed, w0 = ids.copy(), w.copy()
    fixed[1, 2] = 0 if 0 not in fixed[1] else int(np.setdiff1d(np.arange(E), fixed[1])[0])
    w0[1, 2] = 0.0
    out_ref, _, _, _ = run_mlp(w4, g, d, x, fixed, w0, w4.MOE_PATH_DECODE)
    assert torch.equal(out_bad.view(torch.int16), out_ref.view(torch.int16))


def test_moe_mlp_decode_in_a_graph(w4):
    # the decode launch captured in a CUDA graph: replays equal the eager call
    T, k, E, H, I = 2, 8, 32, 2048, 768
    ids, w = routing(980, T, k, E)
    g, d = mlp_experts(981, E, H, I, torch.float16)
    x = si.x(si.config_seed(982), T, H).to(DEV)
    ids_d, w_d = torch.from_numpy(ids).to(DEV), torch.from_numpy(w).to(DEV)
    gate_up = w4.MoeExperts(*g, epilogue=w4.EPILOGUE_SILU_MUL, max_slots=T * k)
    down = w4.MoeExperts(*d, max_slots=T * k)
    mlp = w4.MoeMlp(gate_up, down, T, k, path=w4.MOE_PATH_DECODE)
    try:
        eager = mlp(x, ids_d, w_d)
        out = torch.empty_like(eager)
        st = torch.cuda.Stream()
        st.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=st):
            mlp(x, ids_d, w_d, out=out, stream=st)
        for _ in range(3):
            out.zero_()
            graph.replay()
            torch.cuda.synchronize()
            assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    finally:
        mlp.destroy()
        gate_up.destroy()
        down.destroy()


def test_moe_mlp_decode_path_rules(w4):
    # more tokens than the decode kernel takes run the chain (AUTO) or are
    # refused (forced DECODE); a gate+up without SiLU-and-mul never decodes
    E, H, I = 8, 1024, 512
    g, d = mlp_experts(990, E, H, I, torch.float16)
    gate_up = w4.MoeExperts(*g, epilogue=w4.EPILOGUE_SILU_MUL, max_slots=16 * 2)
    down = w4.MoeExperts(*d, max_slots=16 * 2)
    mlp = w4.MoeMlp(gate_up, down, 16, 2)
    try:
        assert mlp.path(8) == w4.MOE_PATH_DECODE
        assert mlp.path(9) == w4.MOE_PATH_CHAIN
        mlp.set_path(w4.MOE_PATH_DECODE)
        with pytest.raises(w4.W4A16Error):
            mlp.path(9)
        mlp.set_path(w4.MOE_PATH_CHAIN)
        assert mlp.path(1) == w4.MOE_PATH_CHAIN
    finally:
        mlp.destroy()
        gate_up.destroy()
        down.destroy()


# (T, k, E, H, I, dtype): the most slots a launch takes (T*k = 128), one
# choice per token, 1024 experts, a one-group intermediate (I 128)
DECODE_EDGE_CASES = [(8, 16, 128, 1024, 512, torch.float16), (8, 1, 4, 1024, 512, torch.float16),
                     (1, 8, 1024, 1024, 256, torch.float16), (4, 4, 16, 1024, 128, torch.float16)]


@pytest.mark.parametrize("T,k,E,H,I,dt", DECODE_EDGE_CASES)
def test_moe_mlp_decode_edge_shapes(w4, T, k, E, H, I, dt):
    seed = 1200 + T * 31 + k * 7 + E + I
    ids, w = routing(seed, T, k, E)
    g, d = mlp_experts(seed + 1, E, H, I, dt)
    x = si.x(si.config_seed(seed, 5), T, H).float().to(dt)
    out, taken, h, o = run_mlp(w4, g, d, x, ids, w, w4.MOE_PATH_DECODE)
    assert taken == w4.MOE_PATH_DECODE
    check_mlp_steps(g, d, x, ids, w, out, h, o, E, f"decode edge T={T} k={k} E={E} I={I}")


def test_moe_mlp_decode_bf16_wide_range(w4):
    # bf16 tokens 2^20 apart in magnitude: each staged row (x, and the
    # intermediate rows) carries its own power-of-two scale
    T, k, E, H, I = 4, 4, 16, 1024, 512
    ids, w = routing(1300, T, k, E)
    g, d = mlp_experts(1301, E, H, I, torch.bfloat16)
    x = si.x(si.config_seed(1302), T, H).float()
    x[1] *= 2.0 ** 20
    x[3] *= 2.0 ** -20
    x = x.to(torch.bfloat16)
    out, _, h, o = run_mlp(w4, g, d, x, ids, w, w4.MOE_PATH_DECODE)
    r_srt, r_pos, _ = oracle.moe_align(ids, E)
    h_ref = oracle.silu_mul(oracle.moe_linear(bits16(x), host(g[0]).view(np.uint32), bits16(g[1]),
                                              host(g[2]).view(np.uint32), ids, dtype="bf16"))[r_srt]
    o_ref = oracle.moe_linear(bits16(h)[r_pos], host(d[0]).view(np.uint32), bits16(d[1]),
                              host(d[2]).view(np.uint32), ids, per_slot=True, dtype="bf16")[r_srt]
    out_ref = oracle.moe_sum(o.double().cpu().numpy()[r_pos], w.astype(np.float64))
    # the rule is relative to each call's largest output: check the rows of
    # each token (and their slots) on their own scale
    tok = (r_srt // k)
    for t in range(T):
        rows = np.where(tok == t)[0]
        assert_close(h[rows], h_ref[rows], f"bf16 wide range: gate+up, token {t}")
        assert_close(o[rows], o_ref[rows], f"bf16 wide range: down, token {t}")
        assert_close(out[t:t + 1], out_ref[t:t + 1], f"bf16 wide range: sum, token {t}")


def test_moe_mlp_decode_varying_tokens_on_one_handle(w4):
    # one handle, calls with 3, 8, 1 and 8 tokens: the counters a call leaves
    # zeroed serve the next, whatever its number of tiles
    E, k, H, I = 32, 8, 1024, 512
    g, d = mlp_experts(1400, E, H, I, torch.float16)
    gate_up = w4.MoeExperts(*g, epilogue=w4.EPILOGUE_SILU_MUL, max_slots=8 * k)
    down = w4.MoeExperts(*d, max_slots=8 * k)
    mlp = w4.MoeMlp(gate_up, down, 8, k, path=w4.MOE_PATH_DECODE)
    try:
        for i, T in enumerate((3, 8, 1, 8)):
            ids, w = routing(1401 + i, T, k, E)
            x = si.x(si.config_seed(1402, i), T, H)
            out = mlp(x.to(DEV), torch.from_numpy(ids).to(DEV), torch.from_numpy(w).to(DEV))
            torch.cuda.synchronize()
            h, o = (t.clone() for t in mlp.intermediates(T * k))
            check_mlp_steps(g, d, x, ids, w, out, h, o, E, f"call {i} T={T}")
    finally:
        mlp.destroy()
        gate_up.destroy()
        down.destroy()


def test_moe_mlp_decode_no_valid_expert(w4):
    # every id outside [0, E): the status bit is set and every output is an
    # empty sum (zero), as on the chain path
    T, k, E, H, I = 2, 4, 8, 1024, 512
    g, d = mlp_experts(1500, E, H, I, torch.float16)
    ids = np.full((T, k), E + 3, dtype=np.int32)
    ids[1, 2] = -1
    w = np.full((T, k), 0.25, dtype=np.float32)
    x = si.x(si.config_seed(1501), T, H)
    for path in (w4.MOE_PATH_DECODE, w4.MOE_PATH_CHAIN):
        out, taken, _, _ = run_mlp(w4, g, d, x, ids, w, path)
        assert taken == path
        assert w4.w4a16_device_status() & 1024
        assert torch.count_nonzero(out.float()) == 0
