"""The ZeRO-3 per-unit gather (copy of a unit's N bf16 shards into a unit
buffer, CMU 15-779 Lecture 13 notes §3.3 and §5.1) against the oracle's
gather, for units whose flat base is not a multiple of 8 (padding to a
multiple of N moves it), destination buffers at every offset from a 16-byte
boundary and ragged unit lengths.  Elements around the destination range
must keep their sentinel values."""

import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from gpu_common import ensure_built, make_problem, oracle_run, run_gpu, to_np

pytestmark = pytest.mark.gpu

SENTINEL = -12345


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


@pytest.mark.parametrize("n", [3, 8, 5])
def test_gather_every_base_and_destination_offset(n):
    sizes = [5, 1, 9, 2, 17, 3, 8 * 300 + 6, 4, 11, 7, 1_000_003, 6, 16]
    pb = make_problem(si.from_units(sizes), n, 3, steps=1, seed=500 + n)
    ref = oracle_run(pb)
    fs = run_gpu(pb, gather_check=False)
    try:
        lay = pb.lay
        for i in range(fs.n_units):
            numel, padded, shard, base = fs.layout(i)
            want = oracle.gather_unit(ref[3], int(base), int(padded), n)
            for o in range(8):
                buf = torch.full((padded + 16,), SENTINEL, dtype=torch.int16, device="cuda")
                fs.gather_weights(i, buf[o:o + padded].view(torch.bfloat16))
                torch.cuda.synchronize()
                got = buf.cpu().numpy()
                assert np.array_equal(got[o:o + padded].view(np.uint16), want), (i, o)
                assert (got[:o] == SENTINEL).all() and (got[o + padded:] == SENTINEL).all(), (i, o)
        # every unit at once (unit -1), into an unaligned buffer
        total = int(lay.total_padded)
        buf = torch.full((total + 16,), SENTINEL, dtype=torch.int16, device="cuda")
        fs.gather_weights(-1, buf[3:3 + total].view(torch.bfloat16))
        torch.cuda.synchronize()
        got = buf.cpu().numpy()
        assert np.array_equal(got[3:3 + total].view(np.uint16), ref[3])
        assert (got[:3] == SENTINEL).all() and (got[3 + total:] == SENTINEL).all()
    finally:
        fs.close()


def test_gather_launch_count():
    # an aligned unit that is a whole number of vectors takes the plain copy;
    # every other unit one launch of the shifted copy (head and tail included)
    pb = make_problem(si.from_units([4096, 4099, 33]), 3, 3, steps=1, seed=510)
    fs = run_gpu(pb, gather_check=False)
    try:
        for i in range(fs.n_units):
            numel, padded, shard, base = fs.layout(i)
            buf = torch.empty(padded, dtype=torch.bfloat16, device="cuda")
            fs.gather_weights(i, buf)
            assert fs.last_launches() == 1
            torch.cuda.synchronize()
            assert torch.equal(buf.view(torch.int16), fs.param16[base:base + padded].view(torch.int16))
    finally:
        fs.close()


@pytest.mark.parametrize("n", [3, 8])
def test_gather_units_matches_oracle(n):
    # several units per launch (the ZeRO-3 prefetch), aligned and shifted
    # units mixed in one launch, each destination at its own offset from a
    # 16-byte boundary; sub-ranges and an empty range
    sizes = [5, 1, 9, 2, 17, 3, 8 * 300 + 6, 4, 11, 7, 1_000_003, 6, 16, 4096, 40_000]
    pb = make_problem(si.from_units(sizes), n, 3, steps=1, seed=520 + n)
    ref = oracle_run(pb)
    fs = run_gpu(pb, gather_check=False)
    try:
        lay = [fs.layout(i) for i in range(fs.n_units)]
        want = [oracle.gather_unit(ref[3], int(base), int(padded), n) for (_, padded, _, base) in lay]
        for first, count in ((0, fs.n_units), (2, 5), (fs.n_units - 1, 1), (4, 0)):
            bufs, views = [], []
            for k in range(count):
                padded = int(lay[first + k][1])
                o = (3 * k + first) % 8
                buf = torch.full((padded + 16,), SENTINEL, dtype=torch.int16, device="cuda")
                bufs.append((buf, o, padded))
                views.append(buf[o:o + padded].view(torch.bfloat16))
            fs.gather_units(first, views)
            assert fs.last_launches() == (1 if count else 0)
            torch.cuda.synchronize()
            for k, (buf, o, padded) in enumerate(bufs):
                got = buf.cpu().numpy()
                assert np.array_equal(got[o:o + padded].view(np.uint16), want[first + k]), (first, k, o)
                assert (got[:o] == SENTINEL).all() and (got[o + padded:] == SENTINEL).all(), (first, k, o)
    finally:
        fs.close()


def test_gather_units_more_than_one_launch():
    # 70 units: batches of 32 units per launch -> 3 launches
    sizes = [(37 * k) % 1000 + 1 for k in range(70)]
    pb = make_problem(si.from_units(sizes), 6, 3, steps=1, seed=530)
    fs = run_gpu(pb, gather_check=False)
    try:
        bufs = [torch.empty(int(fs.layout(i)[1]) + 1, dtype=torch.bfloat16, device="cuda")[1:]
                for i in range(fs.n_units)]
        fs.gather_units(0, bufs)
        assert fs.last_launches() == 3
        torch.cuda.synchronize()
        for i, buf in enumerate(bufs):
            numel, padded, shard, base = fs.layout(i)
            assert torch.equal(buf.view(torch.int16), fs.param16[base:base + padded].view(torch.int16)), i
    finally:
        fs.close()
