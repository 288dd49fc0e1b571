"""moe_expert_ffn rejects a block list it cannot trust, and does no expert work.

The staged entry point takes the padded layout from its caller (for example a
replayed routing record).  A block list with an expert id outside [0, N), one
that is not sorted by expert, or a padded row count that is not a whole number
of blocks sets MOE_DEV_ERR_BAD_BLOCKS in the device status word; no GEMM tile
runs, so the expert outputs keep whatever the caller put there.  A later call
with the valid layout gives the same bits as before.  The bad entry is placed
both among the first 256 blocks and past them (the block pass of the tile
list builder takes four blocks per thread and round).
"""
import numpy as np
import pytest

from synth import workloads as W

pytestmark = pytest.mark.gpu

BAD_BLOCKS = 0x4
FILL = 7.0   # exactly representable in bf16


def _layout(c, T, seed):
    import torch
    import invariant_expert_routing_gb300 as moe
    from tests.gpu_util import dev_bf16
    wl, d = c.wl, "cuda"
    N, k = wl.num_experts, wl.top_k
    h_d = dev_bf16(W.make_h(wl, T, seed=seed), d)
    ws = moe.workspace(c.cfg, T, d)
    moe.moe_clear_device_status(ws)
    idx = torch.empty((T, k), dtype=torch.int32, device=d)
    gates = torch.empty((T, k), dtype=torch.float32, device=d)
    moe.moe_route(c.cfg, h_d, c.wg_d, c.bias_d, idx, gates, None, ws)
    rows, nblk = moe.moe_max_padded_rows(c.cfg, T), moe.moe_max_blocks(c.cfg, T)
    kept = torch.empty(T * k, dtype=torch.uint8, device=d)
    pos = torch.empty(T * k, dtype=torch.int32, device=d)
    srt = torch.empty(rows, dtype=torch.int32, device=d)
    blk = torch.empty(nblk, dtype=torch.int32, device=d)
    npad = torch.zeros(1, dtype=torch.int32, device=d)
    counts = torch.empty(N, dtype=torch.int32, device=d)
    dropped = torch.zeros(1, dtype=torch.int32, device=d)
    moe.moe_dispatch_align(c.cfg, idx, kept, pos, srt, blk, npad, counts, dropped, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    return h_d, srt, blk, npad, ws, rows


def _ffn(c, h_d, srt, blk, npad, ws, rows):
    import torch
    import invariant_expert_routing_gb300 as moe
    from tests.gpu_util import host_bf16
    y = torch.full((rows, c.wl.hidden), FILL, dtype=torch.bfloat16, device="cuda")
    moe.moe_clear_device_status(ws)
    moe.moe_expert_ffn(c.cfg, h_d, c.w13_d, c.w2_d, None, None, srt, blk, npad, y, None, ws)
    torch.cuda.synchronize()
    return moe.moe_get_device_status(ws), host_bf16(y)


@pytest.mark.parametrize("name,T", [("tiny", 40), ("qw", 800)])
def test_bad_block_lists_do_no_expert_work(name, T):
    import torch
    from tests.layer_case import LayerCase
    c = LayerCase(W.WORKLOADS[name])
    N, B = c.wl.num_experts, c.wl.block_size
    h_d, srt, blk, npad, ws, rows = _layout(c, T, seed=11)
    P = int(npad.cpu()[0])
    nb = P // B
    assert nb >= 2
    fill_bits = np.asarray(torch.tensor(FILL, dtype=torch.bfloat16).view(torch.int16).item(), dtype=np.uint16)

    st, y_ref = _ffn(c, h_d, srt, blk, npad, ws, rows)
    assert st == 0
    assert (y_ref[:P] != fill_bits).any()       # the valid layout computes expert rows

    blk_host = blk.cpu().numpy()
    cases = []
    for at in sorted({0, min(nb - 1, 300)}):     # among the first 256 blocks and past them
        bad = blk_host.copy()
        bad[at] = N                                # expert id out of range
        cases.append(("range", bad, P))
    if name == "qw":
        assert nb > 300
    first, last = blk_host[0], blk_host[nb - 1]
    assert first != last
    bad = blk_host.copy()
    bad[0], bad[nb - 1] = last, first              # not sorted by expert
    cases.append(("order", bad, P))
    cases.append(("rows", blk_host.copy(), P - 1))  # not a whole number of blocks

    for what, bad_blk, bad_p in cases:
        b_d = torch.from_numpy(bad_blk).to("cuda")
        p_d = torch.tensor([bad_p], dtype=torch.int32, device="cuda")
        st, y = _ffn(c, h_d, srt, b_d, p_d, ws, rows)
        assert st & BAD_BLOCKS, what
        assert (y == fill_bits).all(), what        # no GEMM tile ran

    st, y_again = _ffn(c, h_d, srt, blk, npad, ws, rows)
    assert st == 0
    assert np.array_equal(y_again[:P], y_ref[:P])
