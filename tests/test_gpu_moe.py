"""GPU parity of the MoE expert FFN in FP4 against the oracle.

"Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs": tokens are
quantized to MXFP4 before the expert dispatch (section 2.A), expert groups are
ragged with precomputed offsets (section 2.C).  Stage-wise gates:
  dispatch       offsets, token order and the gathered bytes are exact;
  rebase         UE4M3 scale x row factor == 2^E of every block (exact);
  up-projection  h (FP32, before quantization) within 1e-3 relative Frobenius
                 of float64 SiLU(X W1_g^T) * (X W1_u^T); the MXFP4 codes of h
                 bit-exact against the oracle quantizer applied to that h;
  down-projection BF16 Y within 1e-3 of the BF16 rounding of float64 h W2^T.
"""
import numpy as np
import pytest

from _helpers import dev, dev_bf16, from_mma_layout, host

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


def _deq_expert(oracle, q, s, st, per, e, rows, cols):
    qe = host(q[e * rows:(e + 1) * rows])
    se = from_mma_layout(host(s[e * per:(e + 1) * per]), rows, cols // 16)
    return oracle.nv_dequantize_f64(qe, se, host(st)[e])


def _padded_rows(offsets):
    """Row index of every dispatched row in the per-group padded scale layout."""
    out = []
    tile = 0
    for g in range(len(offsets) - 1):
        n = offsets[g + 1] - offsets[g]
        out += [tile * 128 + i for i in range(n)]
        tile += (n + 127) // 128
    return np.array(out, dtype=np.int64)


def _run_moe(fq, oracle, T, H, I, E, k, seed, check_rows=None):
    import torch
    from micro_scaled_fp4_gb300 import workloads as W
    x = W.moe_activations(T, H, seed=seed)
    topk = W.moe_routing(tokens=T, experts=E, top_k=k, seed=seed + 1)
    w1 = W.moe_weights_torch(E, 2 * I, H, seed + 2, "cuda")
    w2 = W.moe_weights_torch(E, H, I, seed + 3, "cuda")

    # a1: quantize the tokens once, before dispatch
    q, s = fq.mx_quantize(dev_bf16(x))
    del x
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
    for e in range(E):
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
    e8 = host(d["s"][sel_t]).astype(np.int64) - 127
    recon = oracle.e4m3_values()[ue_rows] * host(rs[sel_t]).astype(np.float64)[:, None]
    assert np.array_equal(recon, np.exp2(np.repeat(e8, 2, axis=1).astype(np.float64)))

    # weights (offline): NVFP4, RNE, per-expert tensor scale
    w1q, w1s, w1t, w1per = _quantize_experts(fq, w1, E, 2 * I, H)
    w2q, w2s, w2t, w2per = _quantize_experts(fq, w2, E, H, I)
    del w1, w2

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

    hq_h, hs_h, hdbg_h = host(hq[sel_t]), host(hs[sel_t]), host(hdbg[sel_t])
    y_h = host(y[sel_t].float())
    # the MXFP4 codes of h are the oracle's quantization of the kernel's FP32 h
    qr, sr = oracle.mx_quantize(hdbg_h)
    assert np.array_equal(hq_h, qr) and np.array_equal(hs_h, sr)

    a_deq = oracle.mx_dequantize_f64(host(d["q"][sel_t]), host(d["s"][sel_t]))
    h_deq = oracle.mx_dequantize_f64(hq_h, hs_h)
    pos = 0
    for e, sel in checks:
        part = slice(pos, pos + sel.size)
        pos += sel.size
        w1d = _deq_expert(oracle, w1q, w1s, w1t, w1per, e, 2 * I, H)
        h_ref = oracle.moe_up_gate(a_deq[part], w1d, I)
        assert oracle.rel_frobenius(hdbg_h[part], h_ref) <= TOL, e
        w2d = _deq_expert(oracle, w2q, w2s, w2t, w2per, e, H, I)
        y_ref = oracle.gemm_ref(h_deq[part], w2d)
        assert oracle.rel_frobenius(y_h[part], _bf16_round(y_ref)) <= TOL, e
    return offs


def test_moe_small(fq, oracle):
    """700 tokens, hidden 512, intermediate 256, top-2 of 8 experts (ragged)."""
    offs = _run_moe(fq, oracle, T=700, H=512, I=256, E=8, k=2, seed=20)
    assert offs[-1] == 1400


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
    d = fq.moe_dispatch(dev(topk), q, s, E)
    rows_ref, offs_ref = oracle.moe_dispatch(topk, E)
    assert np.array_equal(host(d["offsets"]), offs_ref)
    assert np.array_equal(host(d["row_token"]), rows_ref)
    assert np.array_equal(host(d["q"]), host(q)[rows_ref])
    w = W.moe_weights_torch(E, 256, H, 4, "cuda")
    wq, ws, wt, wper = _quantize_experts(fq, w, E, 256, H)
    ue, rs = fq.mx_rebase_scales(d["s"], d["offsets"], H, E)
    y = fq.grouped_gemm(d["q"], ue, rs, wq, ws, wt, d["offsets"], E, 256)
    torch.cuda.synchronize()
    assert fq.fp4q_device_status() == 0
    a_deq = oracle.mx_dequantize_f64(host(d["q"]), host(d["s"]))
    for e in (2, 4):
        lo, hi = offs_ref[e], offs_ref[e + 1]
        ref = oracle.gemm_ref(a_deq[lo:hi], _deq_expert(oracle, wq, ws, wt, wper, e, 256, H))
        assert oracle.rel_frobenius(host(y.float())[lo:hi], _bf16_round(ref)) <= TOL


def test_moe_full_size_sampled(fq, oracle):
    """65536 tokens of hidden 7168, top-8 of 64 experts (Zipf 1.1), expert FFN
    7168 -> 2x2048 (SiLU gate) -> 7168; every stage run at full size, the GEMM
    stages checked on 6 sampled rows of every expert."""
    _run_moe(fq, oracle, T=65536, H=7168, I=2048, E=64, k=8, seed=8, check_rows=6)
