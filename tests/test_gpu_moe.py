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
    # w4a16_moe_mlp (both linears in one expert-MMA launch, down tiles waiting
    # for their gate+up tiles) against the call-by-call chain, which the test
    # above checks against the oracle step by step; run twice (the completion
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
    mlp = w4.MoeMlp(gate_up, down, T, k)
    try:
        outs = [mlp(x, ids_d, w_d) for _ in range(2)]
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
