"""The N>1 path on the CPU: two gloo ranks split the heads of one scan on
group boundaries, each computes its slice (with the oracle, standing in for
one GPU's ssd_scan_fwd), and the assembled result equals the unsplit one.
Also checks the max-over-ranks timing reduction the benchmark uses."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from state_space_model_chunked_gb300.sharding import (batch_range, head_range, head_shard,
                                                      max_over_ranks)


def test_head_ranges_cover_all_heads_on_group_boundaries():
    for H, G in [(80, 1), (24, 4), (32, 8), (6, 3)]:
        for world in (1, 2, 3, 4, 8):
            cuts = [head_range(H, G, world, r) for r in range(world)]
            assert cuts[0][0] == 0 and cuts[-1][1] == H
            for (a0, a1), (b0, b1) in zip(cuts, cuts[1:]):
                assert a1 == b0
            for a0, a1 in cuts:
                assert a0 % (H // G) == 0 and a1 % (H // G) == 0


def test_head_shards_split_a_single_group_on_pair_boundaries():
    for H, G, world in [(80, 1, 2), (80, 1, 4), (80, 1, 8), (24, 1, 4), (32, 2, 4), (48, 2, 8)]:
        cuts = [head_shard(H, G, world, r) for r in range(world)]
        assert cuts[0][0] == 0 and cuts[-1][1] == H
        for a, b in zip(cuts, cuts[1:]):
            assert a[1] == b[0]
        for h0, h1, g0, g1 in cuts:
            assert h1 - h0 == H // world and h0 % 2 == 0
            assert g1 == g0 + 1 and h0 // (H // G) == g0 and (h1 - 1) // (H // G) == g0
    # whole groups when there are enough of them, or when a group cannot split evenly
    assert [head_shard(32, 8, 4, r) for r in range(4)] == \
        [(h0, h1, h0 // 4, h1 // 4) for h0, h1 in (head_range(32, 8, 4, r) for r in range(4))]
    assert [head_shard(6, 1, 4, r) for r in range(4)] == [(0, 0, 0, 0)] * 3 + [(0, 6, 0, 1)]


def test_batch_ranges_partition():
    for batch in (1, 7, 16, 256):
        for world in (1, 2, 4, 8):
            cuts = [batch_range(batch, world, r) for r in range(world)]
            assert sum(b - a for a, b in cuts) == batch
            assert cuts[0][0] == 0 and cuts[-1][1] == batch


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out_dir):
    import torch.distributed as dist

    import oracle
    from state_space_model_chunked_gb300 import inputs as gen
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    H, G = 8, 2
    inp = gen.scan_inputs(2, 96, H, 8, 16, G, "bf16", seed=123, random_init=True)
    h0, h1 = head_range(H, G, world, rank)
    g0, g1 = h0 // (H // G), h1 // (H // G)
    sl = slice(h0, h1)
    # this rank's slice: its heads and the groups they belong to
    y, fin = oracle.scan_seq(inp["x"][:, :, sl], inp["dt"][:, :, sl], inp["A"][sl],
                             inp["B"][:, :, g0:g1], inp["C"][:, :, g0:g1], inp["D"][sl],
                             inp["init"][:, sl], nthreads=1)
    np.save(os.path.join(out_dir, f"y{rank}.npy"), y)
    np.save(os.path.join(out_dir, f"f{rank}.npy"), fin)
    worst = max_over_ranks(float(rank + 1) * 1.5, dist)
    np.save(os.path.join(out_dir, f"t{rank}.npy"), np.array([worst]))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_reassemble_the_scan(tmp_path):
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_worker, args=(r, world, port, str(tmp_path)))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    import oracle
    from state_space_model_chunked_gb300 import inputs as gen
    inp = gen.scan_inputs(2, 96, 8, 8, 16, 2, "bf16", seed=123, random_init=True)
    y_full, f_full = oracle.scan_seq(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                                     inp["D"], inp["init"])
    ys = [np.load(tmp_path / f"y{r}.npy") for r in range(world)]
    fs = [np.load(tmp_path / f"f{r}.npy") for r in range(world)]
    assert oracle.rel_l2(np.concatenate(ys, axis=2), y_full) < 1e-13
    assert oracle.rel_l2(np.concatenate(fs, axis=1), f_full) < 1e-13
    for r in range(world):
        assert float(np.load(tmp_path / f"t{r}.npy")[0]) == 3.0


def test_sequence_ranges_partition_and_balance():
    from state_space_model_chunked_gb300 import inputs as gen
    from state_space_model_chunked_gb300.sharding import sequence_range
    for lengths in ([5, 0, 13, 1, 9], gen.packed_lengths(47, 64, 8192, seed=5), [100], [0, 0]):
        cu = np.concatenate([[0], np.cumsum(lengths)])
        T, longest = int(cu[-1]), max(lengths)
        for world in (1, 2, 3, 4, 8):
            parts = [sequence_range(cu, world, r) for r in range(world)]
            assert parts[0][0] == 0 and parts[-1][1] == len(lengths)
            for (a0, a1, _), (b0, b1, _) in zip(parts, parts[1:]):
                assert a1 == b0
            for s0, s1, off in parts:
                assert off[0] == 0 and off[-1] == cu[s1] - cu[s0]
                assert off[-1] <= T / world + longest


def _varlen_worker(rank, world, port, out_dir):
    import torch.distributed as dist

    import oracle
    from state_space_model_chunked_gb300 import inputs as gen
    from state_space_model_chunked_gb300.sharding import sequence_range
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    inp = gen.varlen_inputs([30, 7, 0, 55, 12, 40], 4, 8, 16, 2, "bf16", seed=9,
                            random_init=True)
    s0, s1, off = sequence_range(inp["cu"], world, rank)
    t0, t1 = int(inp["cu"][s0]), int(inp["cu"][s1])
    y, fin = oracle.scan_varlen(inp["x"][t0:t1], inp["dt"][t0:t1], inp["A"], inp["B"][t0:t1],
                                inp["C"][t0:t1], off, inp["D"], inp["init"][s0:s1])
    np.save(os.path.join(out_dir, f"vy{rank}.npy"), y)
    np.save(os.path.join(out_dir, f"vf{rank}.npy"), fin)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_reassemble_a_packed_batch(tmp_path):
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_varlen_worker, args=(r, world, port, str(tmp_path)))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    import oracle
    from state_space_model_chunked_gb300 import inputs as gen
    inp = gen.varlen_inputs([30, 7, 0, 55, 12, 40], 4, 8, 16, 2, "bf16", seed=9,
                            random_init=True)
    y_full, f_full = oracle.scan_varlen(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                                        inp["cu"], inp["D"], inp["init"])
    ys = [np.load(tmp_path / f"vy{r}.npy") for r in range(world)]
    fs = [np.load(tmp_path / f"vf{r}.npy") for r in range(world)]
    assert ys[0].shape[0] > 0 and ys[1].shape[0] > 0
    np.testing.assert_array_equal(np.concatenate(ys, axis=0), y_full)
    np.testing.assert_array_equal(np.concatenate(fs, axis=0), f_full)


def _group_split_worker(rank, world, port, out_dir):
    import torch.distributed as dist

    import oracle
    from state_space_model_chunked_gb300 import inputs as gen
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # one group of 8 heads, as the 2.7B layer's single group of 80: split in two
    inp = gen.scan_inputs(1, 80, 8, 8, 16, 1, "bf16", seed=321, random_init=True)
    h0, h1, g0, g1 = head_shard(8, 1, world, rank)
    sl = slice(h0, h1)
    y, fin = oracle.scan_seq(inp["x"][:, :, sl], inp["dt"][:, :, sl], inp["A"][sl],
                             inp["B"][:, :, g0:g1], inp["C"][:, :, g0:g1], inp["D"][sl],
                             inp["init"][:, sl], nthreads=1)
    np.save(os.path.join(out_dir, f"gy{rank}.npy"), y)
    np.save(os.path.join(out_dir, f"gf{rank}.npy"), fin)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_split_one_group(tmp_path):
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_group_split_worker, args=(r, world, port, str(tmp_path)))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    import oracle
    from state_space_model_chunked_gb300 import inputs as gen
    inp = gen.scan_inputs(1, 80, 8, 8, 16, 1, "bf16", seed=321, random_init=True)
    y_full, f_full = oracle.scan_seq(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                                     inp["D"], inp["init"])
    ys = [np.load(tmp_path / f"gy{r}.npy") for r in range(world)]
    fs = [np.load(tmp_path / f"gf{r}.npy") for r in range(world)]
    assert ys[0].shape[2] == 4 and ys[1].shape[2] == 4
    assert oracle.rel_l2(np.concatenate(ys, axis=2), y_full) < 1e-13
    assert oracle.rel_l2(np.concatenate(fs, axis=1), f_full) < 1e-13


# ------------------------------------------------ one sequence split by tokens
def test_token_ranges_partition_on_tile_boundaries():
    from state_space_model_chunked_gb300.sharding import token_range
    for L in (1, 127, 128, 129, 1000, 65536):
        for world in (1, 2, 3, 4, 8):
            cuts = [token_range(L, world, r) for r in range(world)]
            assert cuts[0][0] == 0 and cuts[-1][1] == L
            for (a0, a1), (b0, b1) in zip(cuts, cuts[1:]):
                assert a1 == b0 and a0 <= a1
            assert all(a % 128 == 0 for a, _ in cuts)


def _cpu_sequence_ops():
    """CPU stand-ins for the library's scan, range log-decay and state chain
    (fp64, through the oracle's scan), with the package functions'
    signatures."""
    import torch

    import oracle

    def scan(x, dt, A, B, C, D, chunk, init):
        y, fin = oracle.scan_seq(x.numpy(), dt.numpy(), A.numpy(), B.numpy(), C.numpy(),
                                 None if D is None else D.numpy(),
                                 None if init is None else init.numpy(), nthreads=1)
        return torch.from_numpy(y), torch.from_numpy(fin)

    def log_decay(dt, A):
        return torch.from_numpy(A.numpy()[None, :].astype(np.float64) *
                                dt.numpy().astype(np.float64).sum(axis=1))

    def chain(contrib, decays, init):
        c, d = contrib.numpy(), decays.numpy()
        h = np.zeros(c.shape[1:]) if init is None else init.numpy().astype(np.float64)
        out = np.empty(c.shape)
        for r in range(c.shape[0]):
            out[r] = h
            h = np.exp(d[r])[:, :, None, None] * h + c[r]
        return torch.from_numpy(out)

    return scan, log_decay, chain


def _seq_worker(rank, world, port, out_dir, L):
    import torch
    import torch.distributed as dist

    from state_space_model_chunked_gb300 import inputs as gen
    from state_space_model_chunked_gb300.sharding import scan_sequence_sharded, token_range
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    inp = gen.scan_inputs(2, L, 4, 8, 16, 2, "bf16", seed=321, random_init=True)
    t0, t1 = token_range(L, world, rank)
    part = {k: torch.from_numpy(np.ascontiguousarray(inp[k][:, t0:t1], dtype=np.float64))
            for k in ("x", "dt", "B", "C")}
    whole = {k: torch.from_numpy(inp[k].astype(np.float64)) for k in ("A", "D", "init")}
    y, fin = scan_sequence_sharded(part["x"], part["dt"], whole["A"], part["B"], part["C"],
                                   whole["D"], whole["init"], ops=_cpu_sequence_ops())
    np.save(os.path.join(out_dir, f"sy{rank}.npy"), y.numpy())
    np.save(os.path.join(out_dir, f"sf{rank}.npy"), fin.numpy())
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world,L", [(2, 700), (3, 200)])
def test_gloo_ranks_split_one_sequence_by_tokens(tmp_path, world, L):
    """Ranks hold contiguous token ranges of one sequence (with 3 ranks and 2
    tiles, the first range is empty); after the all-gather and the chain,
    their outputs reassemble the unsplit scan and the last rank holds its
    final state."""
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_seq_worker, args=(r, world, port, str(tmp_path), L))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    import oracle
    from state_space_model_chunked_gb300 import inputs as gen
    inp = gen.scan_inputs(2, L, 4, 8, 16, 2, "bf16", seed=321, random_init=True)
    y_full, f_full = oracle.scan_seq(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                                     inp["D"], inp["init"])
    ys = [np.load(tmp_path / f"sy{r}.npy") for r in range(world)]
    assert oracle.rel_l2(np.concatenate(ys, axis=1), y_full) < 1e-12
    assert oracle.rel_l2(np.load(tmp_path / f"sf{world - 1}.npy"), f_full) < 1e-12
