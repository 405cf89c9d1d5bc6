"""fp4q_moe_dispatch_static: the MoE dispatch for callers that cannot allocate.

Some callers cannot give the library a device workspace: a serving process
that fixes its device-memory budget at start-up and treats any later
allocation as a failure, plain C code that only receives device pointers from
the framework that owns the memory, or a latency-sensitive loop where a
cudaMalloc (which can synchronize the device) is not acceptable.  This entry
point keeps its scratch in a fixed-size static device array instead of a
workspace argument.  Its results must equal those of fp4q_moe_dispatch (which
is bit-exact against the oracle), on consecutive calls that reuse the array,
and it must refuse sizes whose scratch would not fit.

The file is named so that pytest collects it last.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fq():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import micro_scaled_fp4_gb300.fp4q as fq
    fq.load()
    return fq


def _inputs(fq, T, H, E, k, seed):
    import torch
    from micro_scaled_fp4_gb300 import workloads as W
    x = W.moe_activations(T, H, seed=seed)
    topk = W.moe_routing(tokens=T, experts=E, top_k=k, seed=seed + 1)
    q, s = fq.mx_quantize(torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda())
    return torch.from_numpy(topk).cuda(), q, s


def _static_dispatch(fq, topk, q, s, E):
    import torch
    T, k = topk.shape
    C = q.shape[1] * 2
    out = {"offsets": torch.full((E + 1,), -1, dtype=torch.int64, device="cuda"),
           "row_token": torch.full((T * k,), -1, dtype=torch.int32, device="cuda"),
           "q": torch.zeros((T * k, C // 2), dtype=torch.uint8, device="cuda"),
           "s": torch.zeros((T * k, C // 32), dtype=torch.uint8, device="cuda")}
    fq.fp4q_moe_dispatch_static(topk, T, k, E, q, s, C, out["offsets"], out["row_token"], out["q"], out["s"])
    return out


def test_static_dispatch_matches_workspace_dispatch_twice(fq):
    """Two calls in a row with different routings and sizes: each equals the
    workspace entry point exactly (offsets, token order, gathered bytes)."""
    import torch
    for T, H, E, k, seed in [(4096, 1024, 64, 8, 31), (1500, 512, 8, 2, 47)]:
        topk, q, s = _inputs(fq, T, H, E, k, seed)
        got = _static_dispatch(fq, topk, q, s, E)
        ref = fq.moe_dispatch(topk, q, s, E)
        torch.cuda.synchronize()
        for key in ("offsets", "row_token", "q", "s"):
            assert torch.equal(got[key], ref[key]), (T, key)


def test_static_dispatch_rejects_sizes_beyond_the_array(fq):
    import torch
    T, k, E = 1 << 20, 8, 64          # needs ~32 MiB of scratch, more than the array
    assert fq.fp4q_moe_dispatch_workspace_bytes(T, k, E) > fq.MOE_DISPATCH_STATIC_SCRATCH_BYTES
    dummy = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(fq.Fp4qError) as e:
        fq.fp4q_moe_dispatch_static(dummy, T, k, E, dummy, dummy, 64, dummy, dummy, dummy, dummy)
    assert e.value.status == 2 and "static array" in str(e.value)
