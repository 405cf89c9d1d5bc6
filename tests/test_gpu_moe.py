"""GPU parity of the MoE expert FFN in FP4 against the oracle.

"Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs": tokens are
quantized to MXFP4 before the expert dispatch (section 2.A), expert groups are
ragged with precomputed offsets (section 2.C).  The reference is the oracle's
own chain from the seeded tokens, routing and weights; stage-wise gates:
  token quantize  the kernel's MXFP4 of X equals the oracle's (exact);
  dispatch        offsets, token order and the gathered bytes are exact;
  rebase          UE4M3 scale x row factor == 2^E of every block (exact);
  weights         the kernel's NVFP4 of every checked expert equals the
                  oracle's (exact);
  up-projection   h (FP32, before quantization) within 1e-3 relative
                  Frobenius of float64 SiLU(X W1_g^T) * (X W1_u^T);
  h requantized   the MXFP4 codes and E8M0 scales the epilogue writes are,
                  bit for bit, the oracle's MXFP4 of the kernel's own FP32 h
                  (captured through h_debug).  The FP32 h itself is not unique
                  -- it depends on the summation order of the K reduction,
                  which the pages leave open, and is gated against float64
                  above -- while the quantization of a given h is;
  down-projection BF16 Y within 1e-3 of the BF16 rounding of float64
                  h_mx W2^T, h_mx the checked MXFP4 of h.
"""
import numpy as np
import pytest

from _helpers import dev, dev_bf16, from_mma_layout, host, rel_frobenius

pytestmark = pytest.mark.gpu

TOL = 1e-3


@pytest.fixture(scope="module")
def fq():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import micro_scaled_fp4_gb300.fp4q as fq
    fq.load()
    return fq


def _bf16_round(y):
    import torch
    return torch.from_numpy(np.asarray(y, dtype=np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def _quantize_experts(fq, w, E, rows, cols):
    """NVFP4 (RNE, no rotation) of each expert's [rows, cols] BF16 weight, scales in
    the MMA layout back to back, one FP32 tensor scale per expert."""
    import torch
    q = torch.empty((E * rows, cols // 2), dtype=torch.uint8, device="cuda")
    per = fq.fp4q_scales_bytes(rows, cols // 16, fq.FP4Q_SCALES_MMA)
    s = torch.empty(E * per, dtype=torch.uint8, device="cuda")
    st = torch.empty(E, dtype=torch.float32, device="cuda")
    wsb = fq.fp4q_nv_quantize_workspace_bytes(rows, cols)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    for e in range(E):
        fq.fp4q_nv_quantize(w[e], rows, cols, cols, 1, 0, 0, fq.FP4Q_RNE, 0, None, None, st.data_ptr() + 4 * e,
                            q.data_ptr() + e * rows * (cols // 2), s.data_ptr() + e * per, fq.FP4Q_SCALES_MMA,
                            ws, wsb)
    return q, s, st, per


def _bits(t):
    """BF16 bit patterns of a torch BF16 tensor (an input, as generated)."""
    import torch
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def _oracle_expert(oracle, fq_q, fq_s, fq_st, per, w_e, e, rows, cols):
    """The oracle's NVFP4 (RNE, no rotation) of expert e's BF16 weights, after
    checking that the kernel's quantization of it is the same; returns the
    float64 dequantized weights."""
    ref = oracle.nv_quantize(w_e)
    assert np.array_equal(host(fq_q[e * rows:(e + 1) * rows]), ref["q"]), e
    assert np.array_equal(from_mma_layout(host(fq_s[e * per:(e + 1) * per]), rows, cols // 16), ref["s"]), e
    assert host(fq_st)[e] == ref["s_t"], e
    return oracle.nv_dequantize_f64(ref["q"], ref["s"], ref["s_t"])


def _assert_requant_exact(oracle, hq, hs, h_f32, what):
    """The epilogue's MXFP4 of h equals the oracle's MX rule applied to the
    kernel's own FP32 h, every code and every scale byte."""
    q_ref, s_ref = oracle.mx_quantize(np.ascontiguousarray(h_f32, dtype=np.float32))
    nq, ns = int(np.count_nonzero(hq != q_ref)), int(np.count_nonzero(hs != s_ref))
    assert nq == 0 and ns == 0, (what, "differing code bytes", nq, "differing scales", ns)


def _padded_rows(offsets):
    """Row index of every dispatched row in the per-group padded scale layout."""
    out = []
    tile = 0
    for g in range(len(offsets) - 1):
        n = offsets[g + 1] - offsets[g]
        out += [tile * 128 + i for i in range(n)]
        tile += (n + 127) // 128
    return np.array(out, dtype=np.int64)


def _run_moe(fq, oracle, T, H, I, E, k, seed, check_rows=None, check_experts=None, requant_all=False):
    import torch
    from micro_scaled_fp4_gb300 import workloads as W
    x = W.moe_activations(T, H, seed=seed)
    topk = W.moe_routing(tokens=T, experts=E, top_k=k, seed=seed + 1)
    w1 = W.moe_weights_torch(E, 2 * I, H, seed + 2, "cuda")
    w2 = W.moe_weights_torch(E, H, I, seed + 3, "cuda")

    # a1: quantize the tokens once, before dispatch
    q, s = fq.mx_quantize(dev_bf16(x))
    qx_r, sx_r = oracle.mx_quantize(x)
    del x
    assert np.array_equal(host(q), qx_r) and np.array_equal(host(s), sx_r)
    # a9: dispatch
    d = fq.moe_dispatch(dev(topk), q, s, E)
    rows_ref, offs_ref = oracle.moe_dispatch(topk, E)
    offs = host(d["offsets"])
    assert np.array_equal(offs, offs_ref)
    assert np.array_equal(host(d["row_token"]), rows_ref)
    idx = torch.from_numpy(rows_ref).cuda()
    assert torch.equal(d["q"], q[idx]) and torch.equal(d["s"], s[idx])
    del idx

    # the rows every later check looks at
    checks = []
    for e in range(E) if check_experts is None else check_experts:
        sel = np.arange(offs[e], offs[e + 1])
        if check_rows is not None and sel.size > check_rows:
            sel = np.sort(np.random.default_rng(e).choice(sel, check_rows, replace=False))
        if sel.size:
            checks.append((e, sel))
    all_sel = np.concatenate([c[1] for c in checks])
    sel_t = torch.from_numpy(all_sel).cuda()

    # rebase of the dispatched rows' E8M0 scales to UE4M3 per 16 + row factor
    viol = torch.zeros(1, dtype=torch.int32, device="cuda")
    ue, rs = fq.mx_rebase_scales(d["s"], d["offsets"], H, E, viol)
    torch.cuda.synchronize()
    assert int(viol.item()) == 0
    prow = _padded_rows(offs)[all_sel]
    ue_h = host(ue)
    nrows_pad = (ue_h.size // 512) // ((H // 16 + 3) // 4) * 128
    ue_rows = from_mma_layout(ue_h, nrows_pad, H // 16)[prow]
    e8 = sx_r[rows_ref[all_sel]].astype(np.int64) - 127
    recon = oracle.e4m3_values()[ue_rows] * host(rs[sel_t]).astype(np.float64)[:, None]
    assert np.array_equal(recon, np.exp2(np.repeat(e8, 2, axis=1).astype(np.float64)))

    # weights (offline): NVFP4, RNE, per-expert tensor scale
    w1q, w1s, w1t, w1per = _quantize_experts(fq, w1, E, 2 * I, H)
    w2q, w2s, w2t, w2per = _quantize_experts(fq, w2, E, H, I)

    # a10: gated up-projection with the SiLU epilogue and MXFP4 requantization
    hq, hs, hdbg = fq.grouped_gemm(d["q"], ue, rs, w1q, w1s, w1t, d["offsets"], E, 2 * I,
                                   fq.FP4Q_EPI_SILU_GATE_MXFP4, h_debug=True)
    # rebase h, a11: down-projection
    viol.zero_()
    ue2, rs2 = fq.mx_rebase_scales(hs, d["offsets"], I, E, viol)
    y = fq.grouped_gemm(hq, ue2, rs2, w2q, w2s, w2t, d["offsets"], E, H)
    torch.cuda.synchronize()
    assert fq.fp4q_device_status() == 0
    assert int(viol.item()) == 0
    if requant_all:
        # the epilogue's MXFP4 of h on every dispatched row, in row chunks
        for r0 in range(0, hq.shape[0], 65536):
            sl = slice(r0, r0 + 65536)
            _assert_requant_exact(oracle, host(hq[sl]), host(hs[sl]), host(hdbg[sl]), ("rows", r0))

    hq_h, hs_h, hdbg_h = host(hq[sel_t]), host(hs[sel_t]), host(hdbg[sel_t])
    y_h = host(y[sel_t].float())
    pos = 0
    for e, sel in checks:
        part = slice(pos, pos + sel.size)
        pos += sel.size
        tok = rows_ref[sel]
        a_deq = oracle.mx_dequantize_f64(qx_r[tok], sx_r[tok])
        w1d = _oracle_expert(oracle, w1q, w1s, w1t, w1per, _bits(w1[e]), e, 2 * I, H)
        h_ref = oracle.moe_up_gate(a_deq, w1d, I)
        del w1d
        assert rel_frobenius(hdbg_h[part], h_ref) <= TOL, e
        _assert_requant_exact(oracle, hq_h[part], hs_h[part], hdbg_h[part], e)
        w2d = _oracle_expert(oracle, w2q, w2s, w2t, w2per, _bits(w2[e]), e, H, I)
        y_ref = oracle.gemm_ref(oracle.mx_dequantize_f64(hq_h[part], hs_h[part]), w2d)
        del w2d
        assert rel_frobenius(y_h[part], _bf16_round(y_ref)) <= TOL, e
    return offs


def test_moe_small(fq, oracle):
    """700 tokens, hidden 512, intermediate 256, top-2 of 8 experts (ragged)."""
    offs = _run_moe(fq, oracle, T=700, H=512, I=256, E=8, k=2, seed=20)
    assert offs[-1] == 1400


@pytest.mark.parametrize("case", range(3))
def test_moe_random_configs(fq, oracle, case):
    """Seeded random MoE configurations (tokens, hidden and intermediate widths
    in multiples of 128, expert count, top-k) through the whole chain, every
    stage checked as in the fixed cases."""
    rng = np.random.default_rng(9000 + case)
    E = int(rng.integers(2, 21))
    T, H, I, k = int(rng.integers(50, 600)), 128 * int(rng.integers(1, 7)), 128 * int(rng.integers(1, 5)), \
        int(rng.integers(1, min(4, E) + 1))
    offs = _run_moe(fq, oracle, T=T, H=H, I=I, E=E, k=k, seed=9100 + case)
    assert offs[-1] == T * k


def test_moe_k_tails(fq, oracle):
    """K = 384 in both grouped GEMMs (a 128-element last stage), 5 experts."""
    offs = _run_moe(fq, oracle, T=300, H=384, I=384, E=5, k=2, seed=30)
    assert offs[-1] == 600


def test_moe_most_experts(fq, oracle):
    """256 experts (the limit), top-2 over 600 tokens: mostly tiny or empty
    groups, all of them computed; the experts with at least 64 rows are checked
    (the h-code comparison allows one flip per 1000 codes of an expert)."""
    from micro_scaled_fp4_gb300 import workloads as W
    T, E, k, seed = 600, 256, 2, 40
    _, offs_ref = oracle.moe_dispatch(W.moe_routing(tokens=T, experts=E, top_k=k, seed=seed + 1), E)
    big = [e for e in range(E) if offs_ref[e + 1] - offs_ref[e] >= 64]
    assert big and np.sum(np.diff(offs_ref) == 0) > 0       # some large groups and some empty ones
    offs = _run_moe(fq, oracle, T=T, H=256, I=128, E=E, k=k, seed=seed, check_experts=big)
    assert offs[-1] == T * k and len(offs) == E + 1


def test_moe_empty_expert(fq, oracle):
    """A routing that leaves experts empty and one expert with a single row."""
    import torch
    from micro_scaled_fp4_gb300 import workloads as W
    T, H, E = 129, 256, 6
    topk = np.zeros((T, 1), dtype=np.int32)
    topk[:, 0] = 2
    topk[5, 0] = 4
    x = W.moe_activations(T, H, seed=3)
    q, s = fq.mx_quantize(dev_bf16(x))
    qx_r, sx_r = oracle.mx_quantize(x)
    assert np.array_equal(host(q), qx_r) and np.array_equal(host(s), sx_r)
    d = fq.moe_dispatch(dev(topk), q, s, E)
    rows_ref, offs_ref = oracle.moe_dispatch(topk, E)
    assert np.array_equal(host(d["offsets"]), offs_ref)
    assert np.array_equal(host(d["row_token"]), rows_ref)
    assert np.array_equal(host(d["q"]), qx_r[rows_ref])
    w = W.moe_weights_torch(E, 256, H, 4, "cuda")
    wq, ws, wt, wper = _quantize_experts(fq, w, E, 256, H)
    ue, rs = fq.mx_rebase_scales(d["s"], d["offsets"], H, E)
    y = fq.grouped_gemm(d["q"], ue, rs, wq, ws, wt, d["offsets"], E, 256)
    torch.cuda.synchronize()
    assert fq.fp4q_device_status() == 0
    a_deq = oracle.mx_dequantize_f64(qx_r[rows_ref], sx_r[rows_ref])
    for e in (2, 4):
        lo, hi = offs_ref[e], offs_ref[e + 1]
        wd = _oracle_expert(oracle, wq, ws, wt, wper, _bits(w[e]), e, 256, H)
        ref = oracle.gemm_ref(a_deq[lo:hi], wd)
        assert rel_frobenius(host(y.float())[lo:hi], _bf16_round(ref)) <= TOL


def test_moe_requant_of_zero_and_tiny_h(fq, oracle):
    """The SiLU-gate epilogue's MXFP4 requantization on the edge cases of the
    MX rule: expert 1 has all-zero weights (tensor scale 0, so every h is a
    signed zero and every block takes E = -127), expert 2 has its first 64
    gate rows zeroed (h = SiLU(+0) * up = +-0 in whole 32-column blocks),
    and experts 3 and 4 have weights scaled by 2e-19 and 1e-18, which puts
    h between the FP32 subnormals and 2^-120, so block exponents clamp at
    -127 while codes stay non-zero.  Every code and scale must be the
    oracle's MX rule of the kernel's FP32 h."""
    import torch
    from micro_scaled_fp4_gb300 import workloads as W
    T, H, I, E, k = 300, 256, 128, 5, 2
    x = W.moe_activations(T, H, seed=60)
    topk = W.moe_routing(tokens=T, experts=E, top_k=k, seed=61)
    w1 = W.moe_weights_torch(E, 2 * I, H, 62, "cuda")
    w1[1].zero_()
    w1[2][:64].zero_()
    w1[3] = (w1[3].float() * 2e-19).to(torch.bfloat16)
    w1[4] = (w1[4].float() * 1e-18).to(torch.bfloat16)
    q, s = fq.mx_quantize(dev_bf16(x))
    d = fq.moe_dispatch(dev(topk), q, s, E)
    ue, rs = fq.mx_rebase_scales(d["s"], d["offsets"], H, E)
    w1q, w1s, w1t, w1per = _quantize_experts(fq, w1, E, 2 * I, H)
    hq, hs, hdbg = fq.grouped_gemm(d["q"], ue, rs, w1q, w1s, w1t, d["offsets"], E, 2 * I,
                                   fq.FP4Q_EPI_SILU_GATE_MXFP4, h_debug=True)
    torch.cuda.synchronize()
    assert fq.fp4q_device_status() == 0
    offs = host(d["offsets"])
    hq_h, hs_h, h_h = host(hq), host(hs), host(hdbg)
    for e in range(E):
        lo, hi = offs[e], offs[e + 1]
        assert hi > lo, e
        _assert_requant_exact(oracle, hq_h[lo:hi], hs_h[lo:hi], h_h[lo:hi], e)
    # the cases the test is for actually occur
    zero = lambda a: (a.view(np.uint32) & 0x7FFFFFFF) == 0
    e1 = slice(offs[1], offs[2])
    assert np.all(zero(h_h[e1])) and np.all(hs_h[e1] == 0)
    e2 = slice(offs[2], offs[3])
    assert np.all(zero(h_h[e2][:, :64])) and np.all(hs_h[e2][:, :2] == 0)
    assert np.any(np.signbit(h_h[e2][:, :64])) and np.any(~np.signbit(h_h[e2][:, :64]))
    assert np.any((hq_h[e2][:, :32] & 0x88) != 0)          # -0 codes (8) among the zero blocks
    tiny = np.concatenate([h_h[offs[3]:offs[5]]])
    assert np.any((tiny.view(np.uint32) & 0x7F800000) == 0)                   # FP32 subnormal h
    blocks_amax = np.abs(tiny).reshape(tiny.shape[0], -1, 32).max(axis=2)
    clamped = (blocks_amax > 0) & (blocks_amax < 2.0 ** -125)
    assert clamped.sum() > 0 and np.all(hs_h[offs[3]:offs[5]][clamped] == 0)
    q_t = hq_h[offs[3]:offs[5]].reshape(tiny.shape[0], -1, 16)[clamped]
    assert np.any((q_t & 0x77) != 0)                        # non-zero codes under the clamp


def test_moe_full_size(fq, oracle):
    """65536 tokens of hidden 7168, top-8 of 64 experts (Zipf 1.1), expert FFN
    7168 -> 2x2048 (SiLU gate) -> 7168, every stage at full size.  Token
    quantization, dispatch (offsets, token order, gathered bytes) and the
    epilogue's MXFP4 of h are compared on all 524288 dispatched rows; the
    GEMM stages (h against float64, Y) and the experts' NVFP4 weights on 24
    sampled rows of every non-empty expert."""
    _run_moe(fq, oracle, T=65536, H=7168, I=2048, E=64, k=8, seed=8, check_rows=24, requant_all=True)


@pytest.mark.parametrize("cols_seq", [(7168,), (2048, 128), (32768, 16384, 32768), (33024,)])
def test_mx_rebase_scales_exact(fq, oracle, cols_seq):
    """fp4q_mx_rebase_scales against the oracle's rebase on every grouped row:
    the UE4M3 bytes (read back through the padded MMA layout), the FP32 row
    factors bit for bit, and the violation count.  Ragged groups (empty, 1,
    127-129, 255, 256 and 300 rows), rows past offsets[groups] that must be
    ignored, all-zero rows, the largest E8M0 byte and planted blocks just
    inside (E - B = -9) and outside (-10) the representable range.  cols 128
    is the narrowest tile form (one 32-bit word per row), 32768 the widest
    (132 KB of shared memory, run again after a narrower one), 33024 takes the
    row-wise kernel."""
    import torch
    sizes = [0, 1, 127, 128, 129, 0, 255, 256, 300, 2]
    G = len(sizes)
    offs = np.zeros(G + 1, dtype=np.int64)
    offs[1:] = np.cumsum(sizes)
    n = int(offs[-1])
    R = n + 5                                              # 5 rows past the last group
    for cols in cols_seq:
        S32 = cols // 32
        rng = np.random.default_rng(cols)
        s = rng.integers(110, 140, (R, S32), dtype=np.uint8)
        s[rng.random((R, S32)) < 0.02] = 0
        s[3] = 0                                           # all-zero row
        s[7, 0] = 254
        for r in range(10, n, 37):                         # E - B = -9 and -10 beside the row max
            s[r, :] = 130
            s[r, -1] = 130 - 17
            if S32 > 2:
                s[r, 1] = 130 - 18
        ue_ref, f_ref, v_ref = oracle.mx_rebase_scales(s[:n])
        viol = torch.zeros(1, dtype=torch.int32, device="cuda")
        ue, rs = fq.mx_rebase_scales(dev(s), dev(offs), cols, G, viol)
        torch.cuda.synchronize()
        S16 = cols // 16
        ue_h = host(ue)
        nrows_pad = (ue_h.size // 512) // ((S16 + 3) // 4) * 128
        got = from_mma_layout(ue_h, nrows_pad, S16)[_padded_rows(offs)]
        assert np.array_equal(got, ue_ref), cols
        assert np.array_equal(host(rs)[:n].view(np.uint32), f_ref.view(np.uint32)), cols
        assert int(viol.item()) == v_ref and v_ref > 0, cols


@pytest.mark.parametrize("cols", [2048, 33024])
def test_mx_rebase_scales_clamps_malformed_offsets(fq, oracle, cols):
    """Offsets that decrease or run past `rows` are clamped, each into
    [previous offset, rows]: the call writes nothing past
    fp4q_rebased_scales_bytes (a canary follows the output) and the rows of
    the clamped groups are rebased as with those offsets."""
    import torch
    R, G = 350, 4
    bad = np.array([0, 300, 100, 400, 50], dtype=np.int64)
    clamped = np.array([0, 300, 300, 350, 350], dtype=np.int64)
    s = np.random.default_rng(5).integers(110, 140, (R, cols // 32), dtype=np.uint8)
    size = fq.fp4q_rebased_scales_bytes(R, cols, G)
    out = torch.full((size + 8192,), 0xAB, dtype=torch.uint8, device="cuda")
    rs = torch.zeros(R + 64, dtype=torch.float32, device="cuda")
    rs[R:] = 7.0
    fq.fp4q_mx_rebase_scales(dev(s), R, cols, dev(bad), G, out, rs, None, None)
    torch.cuda.synchronize()
    out_h = host(out)
    assert np.all(out_h[size:] == 0xAB) and np.all(host(rs)[R:] == 7.0)
    S16 = cols // 16
    nrows_pad = (size // 512) // ((S16 + 3) // 4) * 128
    got = from_mma_layout(out_h[:size], nrows_pad, S16)[_padded_rows(clamped)]
    ue_ref, f_ref, _ = oracle.mx_rebase_scales(s)
    assert np.array_equal(got, ue_ref)
    assert np.array_equal(host(rs)[:R].view(np.uint32), f_ref.view(np.uint32))


def test_grouped_gemm_clamps_malformed_offsets(fq):
    """Offsets that decrease or run past `rows` are clamped by the grouped GEMM
    as by the rebase (each into [previous offset, rows]): both epilogues write
    nothing past their outputs (canaries follow D, the h scales and h_debug)
    and give, bit for bit, the results of the clamped offsets."""
    import torch
    from micro_scaled_fp4_gb300 import workloads as W
    R, H, N, G = 350, 256, 256, 4
    bad = np.array([0, 300, 100, 400, 50], dtype=np.int64)
    clamped = np.array([0, 300, 300, 350, 350], dtype=np.int64)
    q, s = fq.mx_quantize(dev_bf16(W.moe_activations(R, H, seed=70)))
    w = W.moe_weights_torch(G, N, H, 71, "cuda")
    wq, ws, wt, _ = _quantize_experts(fq, w, G, N, H)
    CAN = 4096

    def run(offs, epi):
        o = dev(offs)
        ue = torch.zeros(fq.fp4q_rebased_scales_bytes(R, H, G), dtype=torch.uint8, device="cuda")
        rs = torch.zeros(R, dtype=torch.float32, device="cuda")
        fq.fp4q_mx_rebase_scales(s, R, H, o, G, ue, rs, None, None)
        if epi == fq.FP4Q_EPI_STORE_BF16:
            d = torch.full((R * N * 2 + CAN,), 0xAB, dtype=torch.uint8, device="cuda")
            fq.fp4q_grouped_gemm(q, ue, rs, wq, ws, wt, o, R, G, N, H, epi, d, None, None, None)
            torch.cuda.synchronize()
            return [d]
        d = torch.full((R * (N // 4) + CAN,), 0xAB, dtype=torch.uint8, device="cuda")
        hs = torch.full((R * (N // 64) + CAN,), 0xAB, dtype=torch.uint8, device="cuda")
        hd = torch.full((R * (N // 2) + CAN // 4,), 7.0, dtype=torch.float32, device="cuda")
        fq.fp4q_grouped_gemm(q, ue, rs, wq, ws, wt, o, R, G, N, H, epi, d, hs, hd, None)
        torch.cuda.synchronize()
        return [d, hs, hd]

    for epi in (fq.FP4Q_EPI_STORE_BF16, fq.FP4Q_EPI_SILU_GATE_MXFP4):
        got, ref = run(bad, epi), run(clamped, epi)
        assert fq.fp4q_device_status() == 0
        for g_t, r_t in zip(got, ref):
            g_h, r_h = host(g_t), host(r_t)
            tail = g_h.size - (CAN // 4 if g_h.dtype == np.float32 else CAN)
            canary = np.float32(7.0) if g_h.dtype == np.float32 else 0xAB
            assert np.all(g_h[tail:] == canary) and np.all(r_h[tail:] == canary), epi
            assert np.array_equal(g_h[:tail].view(np.uint8), r_h[:tail].view(np.uint8)), epi
