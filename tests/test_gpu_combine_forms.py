"""The combine's launch forms give the same bits.

The combine runs one of several kernels by batch shape: a row split over
several CTAs for a few tokens, one CTA per token (8 features per thread
when H is a multiple of 2048, else 4), and one warp per token for batches
of at least 2048 tokens with 4 to 16 slots.  Each forms every output
feature as h + (fma chain over the kept slots in ascending order, then the
shared expert's row), so a token's output row must not depend on which
form ran.  Here the same token rows are combined in a batch large enough
for the warp form and in smaller prefixes of it that take the other forms;
the rows they share must be bit-identical, dropped and out-of-range slots
included.  (Layer-level parity with the oracle is in test_gpu_parity and
test_gpu_fullsize.)
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("H,k,shared", [(2048, 8, False), (7168, 8, True), (4096, 4, False), (1152, 16, True)])
def test_combine_forms_bit_identical(H, k, shared):
    import torch
    import invariant_expert_routing_gb300 as moe
    from tests.gpu_util import dev_bf16
    from synth import f32_to_bf16
    T = 2048
    cfg = dict(hidden=H, num_experts=64, top_k=k, intermediate=256, block_size=16)
    # positions valid for the smallest prefix below, so every form keeps the
    # same slots
    rows = moe.moe_max_padded_rows(cfg, 16)
    rng = np.random.default_rng(H + k)
    h = f32_to_bf16(rng.standard_normal((T, H)).astype(np.float32))
    y = f32_to_bf16(rng.standard_normal((rows, H)).astype(np.float32))
    pos = rng.integers(0, rows, size=(T, k)).astype(np.int32)
    kept = (rng.random((T, k)) > 0.15).astype(np.uint8)          # dropped routes
    pos[rng.random((T, k)) < 0.05] = -1                             # no row
    gate = rng.random((T, k)).astype(np.float32)
    h_d, y_d = dev_bf16(h), dev_bf16(y)
    ys_d = dev_bf16(f32_to_bf16(rng.standard_normal((T, H)).astype(np.float32))) if shared else None
    pos_d = torch.from_numpy(pos).cuda()
    kept_d = torch.from_numpy(kept).cuda()
    gate_d = torch.from_numpy(gate).cuda()
    outs = {}
    for n in (T, T - 1, 300, 16):
        out = torch.empty((n, H), dtype=torch.bfloat16, device="cuda")
        moe.moe_combine(cfg, h_d[:n], gate_d[:n], kept_d[:n], pos_d[:n], y_d,
                        None if ys_d is None else ys_d[:n], out)
        torch.cuda.synchronize()
        outs[n] = out.view(torch.int16).cpu().numpy()
    for n in (T - 1, 300, 16):
        assert np.array_equal(outs[T][:n], outs[n]), f"rows differ between T={T} and T={n}"
