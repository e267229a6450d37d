"""Output-partitioned layer, host side, on CPU: the column blocks of the
ranks tile the output exactly in whole 128-column tiles, fp4moe_forward_cols
refuses other ranges before any device work, and tp_forward's all-reduce
over two gloo ranks assembles the blocks (a stand-in layer computes each
rank's block on the CPU)."""
import ctypes
import multiprocessing as mp
import os
import socket
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent


@pytest.mark.parametrize("H,world", [(7168, 1), (7168, 2), (7168, 8), (7168, 56), (512, 3), (2304, 5)])
def test_column_blocks_tile_the_output(H, world):
    from block_scaled_fp4_sigmoid_gb300.layer import column_block
    blocks = [column_block(H, r, world) for r in range(world)]
    assert blocks[0][0] == 0 and blocks[-1][1] == H
    for (a0, a1), (b0, b1) in zip(blocks, blocks[1:]):
        assert a1 == b0  # contiguous, disjoint
    widths = [h1 - h0 for h0, h1 in blocks]
    assert all(w > 0 and w % 128 == 0 for w in widths)
    assert max(widths) - min(widths) <= 128  # as even as whole tiles allow


def test_column_block_limits():
    from block_scaled_fp4_sigmoid_gb300.layer import column_block
    with pytest.raises(ValueError):
        column_block(512, 0, 5)  # more ranks than 128-column tiles
    with pytest.raises(ValueError):
        column_block(512, 2, 2)


def test_forward_cols_refuses_bad_ranges_without_a_gpu():
    import block_scaled_fp4_sigmoid_gb300 as fm
    lib = fm.lib()
    d = fm.make_dims(4, 256, 128, 8, 2)
    w = fm.Weights()
    buf = ctypes.create_string_buffer(1024)
    for h0, h1 in ((0, 64), (64, 256), (128, 128), (256, 128), (0, 384), (-128, 128)):
        assert lib.fp4moe_forward_cols(ctypes.byref(d), ctypes.byref(w), buf, buf, h0, h1, None, buf, 1024,
                                       None) == 2, (h0, h1)


def test_forward_cols_paired_down_weights_need_whole_slabs():
    """With the down weights in the row-tile-paired layout (packed = 3) a
    column block must cover whole 256-row slabs; an unknown packing level is
    an invalid argument.  Both are refused before any device work."""
    import block_scaled_fp4_sigmoid_gb300 as fm
    lib = fm.lib()
    d = fm.make_dims(4, 512, 128, 8, 2)
    buf = ctypes.create_string_buffer(4096)
    p = ctypes.addressof(buf)
    w = fm.Weights(p, p, p, p, None, None, None, None, None, None, p, p, 3)
    big = 1 << 40  # the workspace size is only compared before any device work
    for h0, h1 in ((128, 512), (0, 384), (256, 384)):
        assert lib.fp4moe_forward_cols(ctypes.byref(d), ctypes.byref(w), buf, buf, h0, h1, None, buf, big,
                                       None) == 2, (h0, h1)
    w.packed = 4
    assert lib.fp4moe_forward_cols(ctypes.byref(d), ctypes.byref(w), buf, buf, 0, 512, None, buf, big, None) == 1
    w.packed = 3
    d3 = fm.make_dims(4, 384, 128, 8, 2)  # H not a multiple of 256
    assert lib.fp4moe_forward(ctypes.byref(d3), ctypes.byref(w), buf, buf, None, buf, big, None) == 2


class _StandIn:
    """The interface tp_forward uses: dims.H and forward_cols (here on the
    CPU: the block's columns of 2x, zero elsewhere)."""

    def __init__(self, H):
        from types import SimpleNamespace
        self.dims = SimpleNamespace(H=H)
        self.column_unit = 128

    def forward_cols(self, x, h0, h1):
        import torch
        out = torch.zeros_like(x)
        out[:, h0:h1] = 2 * x[:, h0:h1]
        return out


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, str(ROOT))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist

    from block_scaled_fp4_sigmoid_gb300.layer import tp_forward
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x = torch.arange(3 * 640, dtype=torch.float32).reshape(3, 640)
        out = tp_forward(_StandIn(640), x)
        q.put((rank, bool(torch.equal(out, 2 * x))))
    finally:
        dist.destroy_process_group()


def test_tp_forward_assembles_the_blocks_on_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        results = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [p.exitcode for p in procs] == [0, 0]
    assert results == [(0, True), (1, True)]
