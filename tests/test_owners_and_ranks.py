"""Owner assignment (host planner vs oracle, validity, bounds) and the multi-rank host
logic on CPU: two gloo ranks compute the same owner plan, and the bench's timing
reduction takes the slowest rank."""
import itertools
import os
import sys

import numpy as np
import pytest

from oracle import muon_ref as ref
from muon_optimizer_step_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_ns_cost_matches_printed_count():
    # One 256 x 128 matrix, 5 iterations: 73.4 MFLOP with symmetric Gram and A^2.
    assert ref.ns_cost(256, 128, 5) == 73_400_320
    assert ref.ns_cost(128, 256, 5) == ref.ns_cost(256, 128, 5)


@pytest.mark.parametrize("wl_name,n_shards", [("llama3_8b_8shards", 8), ("ragged_small", 3),
                                              ("ragged_small", 8), ("gpt2_small_x12", 4),
                                              ("moe_64e", 5), ("single_256x128", 2)])
def test_owner_plan_valid_and_matches_oracle(wl_name, n_shards):
    capi = pytest.importorskip("muon_optimizer_step_gb300.capi")
    wl = inputs.WORKLOADS[wl_name]
    lay = capi.muon_layout_create(wl.shapes, n_shards, 0, wl.is_matrix)
    owner, cost = capi.muon_assign_owners(lay, 5)
    o = ref.flat_layout(wl.shapes, n_shards, wl.is_matrix)
    owner_or, cost_or = ref.assign_owners(o, 5)
    assert owner == owner_or
    np.testing.assert_allclose(cost, cost_or, rtol=0, atol=0)
    for i in range(len(wl.shapes)):
        if not wl.is_matrix[i]:
            assert owner[i] == -1
            continue
        cands = ref.shards_of(o, i)
        assert owner[i] in cands
        if len(cands) == 1:
            assert owner[i] == cands[0]  # unsharded matrices are computed locally


def _makespan(owner, layout, n):
    load = [0.0] * n
    for i, (r, c) in enumerate(layout["shapes"]):
        if layout["is_matrix"][i]:
            load[owner[i]] += ref.ns_cost(r, c)
    return max(load)


@pytest.mark.parametrize("seed", range(6))
def test_owner_plan_against_brute_force(seed):
    rng = np.random.default_rng(seed)
    shapes = [(int(rng.integers(1, 40)), int(rng.integers(1, 40))) for _ in range(6)]
    n = 2 + seed % 2
    o = ref.flat_layout(shapes, n)
    owner, load = ref.assign_owners(o)
    cands = [ref.shards_of(o, i) for i in range(len(shapes))]
    best = min(_makespan(list(choice), o, n) for choice in itertools.product(*cands))
    assert _makespan(owner, o, n) >= best
    # Without shard restrictions (every matrix eligible everywhere) LPT is within
    # Graham's 4/3 - 1/(3n) of the optimum.
    free_load = [0.0] * n
    jobs = sorted((ref.ns_cost(r, c) for r, c in shapes), reverse=True)
    for j in jobs:
        free_load[int(np.argmin(free_load))] += j
    opt = min(max(sum(ref.ns_cost(*shapes[i]) for i in range(len(shapes)) if a[i] == k)
                  for k in range(n)) for a in itertools.product(range(n), repeat=len(shapes)))
    assert max(free_load) <= (4 / 3 - 1 / (3 * n)) * opt + 1e-9


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from muon_optimizer_step_gb300 import capi, inputs as inp
    import bench
    wl = inp.WORKLOADS["llama3_8b_8shards"]
    lay = capi.muon_layout_create(wl.shapes, 8, 0, wl.is_matrix)
    owner, _ = capi.muon_assign_owners(lay, 5)
    mine = torch.tensor(owner, dtype=torch.int64)
    got = [torch.zeros_like(mine) for _ in range(world)]
    dist.all_gather(got, mine)
    agree = all(torch.equal(g, got[0]) for g in got)
    # bench's timing rule: every rank reports the slowest rank's times
    red = bench.reduce_max_over_ranks([1.0 + rank, 10.0 - rank], dist, "cpu")
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{int(agree)} {red[0]} {red[1]}\n")
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_owner_plan_and_max_timing(tmp_path):
    pytest.importorskip("muon_optimizer_step_gb300.capi")
    import torch.multiprocessing as mp
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn")
    for r in range(2):
        agree, a, b = open(tmp_path / f"rank{r}.txt").read().split()
        assert agree == "1"
        assert float(a) == 2.0 and float(b) == 10.0


def _rank_dies_main(rank, world, port, out_dir, timeout_s):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import datetime
    import time
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=timeout_s))
    import bench
    if rank == 1:
        # Leaves between steps: never joins the timing reduction.
        os._exit(0)
    t0 = time.monotonic()
    try:
        bench.reduce_max_over_ranks([1.0], dist, "cpu")
        outcome = "returned"
    except Exception as e:  # the surviving rank must get an error, not hang
        outcome = "error:" + type(e).__name__
    with open(os.path.join(out_dir, "rank0.txt"), "w") as f:
        f.write(f"{outcome} {time.monotonic() - t0:.3f}\n")
    os._exit(0)


def test_surviving_rank_gets_an_error_when_a_rank_dies(tmp_path):
    """Failure detection on the host: one of two gloo ranks exits instead of joining the
    step-time reduction; the other's collective fails within the process-group timeout
    instead of waiting forever (bench.py sets such a timeout on its NCCL group)."""
    import torch.multiprocessing as mp
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    timeout_s = 10
    mp.start_processes(_rank_dies_main, args=(2, port, str(tmp_path), timeout_s), nprocs=2,
                       start_method="spawn")
    outcome, elapsed = open(tmp_path / "rank0.txt").read().split()
    assert outcome.startswith("error:"), outcome
    assert float(elapsed) < 3 * timeout_s
    import bench
    assert 60 <= bench.PG_TIMEOUT_S <= 3600


def test_bench_flop_and_byte_models():
    """bench.py's roofline arithmetic: symmetric and dense Newton-Schulz flop counts of a
    single matrix (tall and wide give the same count), the streaming byte model, and the
    traffic record's code digest ignoring comments."""
    import bench
    sym, dense = bench.ns_flops([(256, 128)], [True], 5)
    m, n = 128, 256
    assert sym == 5 * (3 * m * m * n + m ** 3)
    assert dense == 5 * (4 * m * m * n + 2 * m ** 3)
    assert bench.ns_flops([(128, 256)], [True], 5) == (sym, dense)
    assert bench.ns_flops([(128, 256)], [False], 5) == (0, 0)
    assert bench.elementwise_bytes(10, "bf16") == (140, 100)
    assert bench.elementwise_bytes(10, "fp32") == (160, 120)
    assert bench.elementwise_bytes(10, "split") == (180, 140)
    d = bench._ns_sources_sha256()
    assert len(d) == 64 and d == bench._ns_sources_sha256()


def _rank_mem_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    need = 10 ** 9
    both = bench.host_memory_allows(need, world, dist, "cpu", available=100 * need)
    # one rank sees too little: nobody pins
    one = bench.host_memory_allows(need, world, dist, "cpu",
                                   available=100 * need if rank == 0 else 5 * need)
    # room for one rank's buffers but not for both
    tight = bench.host_memory_allows(need, world, dist, "cpu", available=4 * need)
    with open(os.path.join(out_dir, f"mem{rank}.txt"), "w") as f:
        f.write(f"{int(both)} {int(one)} {int(tight)}\n")
    dist.destroy_process_group()


def test_ranks_agree_on_pinning_host_memory(tmp_path):
    """The e2e measurement pins host memory on every rank of one host: the ranks decide
    together, with room for all of them, so that N ranks cannot exhaust the host."""
    import torch.multiprocessing as mp
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mp.start_processes(_rank_mem_main, args=(2, port, str(tmp_path)), nprocs=2,
                       start_method="spawn")
    for r in range(2):
        assert open(tmp_path / f"mem{r}.txt").read().split() == ["1", "0", "0"]
