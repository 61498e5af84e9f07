"""The owner exchange plan ("Add initial Muon+M-FSDPv2 implementation", "Opt step" steps 3
and 5): per rank, the runs of matrix elements sent to owners and received from shard
holders.  Host only: the library's planner is checked by brute force on tiny layouts, and
moving the data with the package's OwnerExchange (torch.distributed point-to-point on CPU
tensors: gloo, 2 and 3 ranks) rebuilds, bit for bit, what the oracle's gather gives on
each owner and, on the way back, what its scatter gives on each shard."""
import os
import socket
import sys

import numpy as np
import pytest

from oracle import muon_ref as ref
from muon_optimizer_step_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
capi = pytest.importorskip("muon_optimizer_step_gb300.capi",
                           reason="libmuon.so not built (run __graft_entry__.build())")


def _layouts():
    rng = np.random.default_rng(7)
    out = []
    for S in (1, 2, 3, 5):
        shapes = [(int(rng.integers(1, 40)), int(rng.integers(1, 40))) for _ in range(9)]
        flags = [bool(rng.random() < 0.8) for _ in shapes]
        owner = [int(rng.integers(0, S)) if f else -1 for f in flags]
        out.append((shapes, flags, S, owner))
    wl = inputs.WORKLOADS["ragged_small"]
    lay = capi.muon_layout_create(wl.shapes, 3, 0, wl.is_matrix)
    out.append((list(wl.shapes), list(wl.is_matrix), 3, capi.muon_assign_owners(lay)[0]))
    return out


@pytest.mark.parametrize("case", range(5))
def test_runs_cover_every_matrix_element_once(case):
    shapes, flags, S, owner = _layouts()[case]
    lay = capi.muon_layout_create(shapes, S, 0, flags)
    o = ref.flat_layout(shapes, S, flags)
    L = o["L"]
    seen_src = {}
    seen_dst = {}
    owned = []
    for r in range(S):
        sends, recvs, numel, offs = capi.muon_exchange_plan(lay, owner, r)
        owned.append(numel)
        for x in sends:
            assert x["src_rank"] == r and x["dst_rank"] == owner[x["param"]]
        for x in recvs:
            assert x["dst_rank"] == r
        # ordering: (peer, parameter, offset)
        keys = [(x["dst_rank"], x["param"], x["shard_off"]) for x in sends]
        assert keys == sorted(keys)
        keys = [(x["src_rank"], x["param"], x["owner_off"]) for x in recvs]
        assert keys == sorted(keys)
        for x in recvs:
            i = x["param"]
            for e in range(x["len"]):
                g = x["src_rank"] * L + x["shard_off"] + e      # flat index of the element
                local = g - o["offsets"][i]                      # its place in the matrix
                assert 0 <= local < shapes[i][0] * shapes[i][1]
                assert x["owner_off"] + e == offs[i] + local
                assert (i, local) not in seen_dst
                seen_dst[(i, local)] = r
        for x in sends:
            for e in range(x["len"]):
                seen_src[(x["param"], x["src_rank"] * L + x["shard_off"] + e)] = r
    # every element of every matrix exactly once, on its owner, taken from its own shard
    for i, (rr, cc) in enumerate(shapes):
        if not flags[i]:
            continue
        for local in range(rr * cc):
            assert seen_dst[(i, local)] == owner[i]
            g = o["offsets"][i] + local
            assert seen_src[(i, g)] == g // L
    assert len(seen_dst) == sum(r * c for (r, c), f in zip(shapes, flags) if f)
    # packed buffers: each owner's parameters back to back at multiples of 4
    for r in range(S):
        _, _, numel, offs = capi.muon_exchange_plan(lay, owner, r)
        mine = [i for i, f in enumerate(flags) if f and owner[i] == r]
        pos = 0
        for i in mine:
            pos = -(-pos // 4) * 4
            assert offs[i] == pos
            pos += shapes[i][0] * shapes[i][1]
        assert numel == pos


def test_sender_and_receiver_lists_pair_up():
    shapes, flags, S, owner = _layouts()[3]
    lay = capi.muon_layout_create(shapes, S, 0, flags)
    plans = [capi.muon_exchange_plan(lay, owner, r) for r in range(S)]
    for s in range(S):
        for d in range(S):
            a = [x for x in plans[s][0] if x["dst_rank"] == d]
            b = [x for x in plans[d][1] if x["src_rank"] == s]
            assert a == b


def test_plan_rejects_bad_owner_and_rank():
    lay = capi.muon_layout_create([(4, 4), (3, 1)], 2, 0, [True, False])
    with pytest.raises(capi.MuonError):
        capi.muon_exchange_plan(lay, [2, -1], 0)
    with pytest.raises(capi.MuonError):
        capi.muon_exchange_plan(lay, [0, -1], 2)
    s, r, n, offs = capi.muon_exchange_plan(lay, [1, 99], 1)  # non-matrix owner ignored
    assert n == 16 and offs == [0, -1]


def _exchange_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    from muon_optimizer_step_gb300 import capi as c
    from muon_optimizer_step_gb300 import inputs as inp
    from muon_optimizer_step_gb300.exchange import OwnerExchange
    from oracle import muon_ref as oref
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # straddling parameters: the ragged set plus a vector, split over `world` shards
    wl = inp.WORKLOADS["ragged_small"]
    shapes = list(wl.shapes) + [(1000, 1), (97, 113)]
    flags = list(wl.is_matrix) + [False, True]
    lay = c.muon_layout_create(shapes, world, 0, flags)
    owner, _ = c.muon_assign_owners(lay)
    ex = OwnerExchange(lay, owner, rank)
    o = oref.flat_layout(shapes, world, flags)
    flat = np.random.default_rng(11).normal(size=lay.numel).astype(np.float32)
    my_shard = torch.from_numpy(oref.shard_flat(flat, o)[rank].astype(np.float32))
    # step 3: shards -> owners
    owned = ex.gather_to_owners(dist, my_shard).numpy()
    full = oref.gather_full(oref.shard_flat(flat, o), o)
    offs = ex.owned_offsets
    ok_gather = all(np.array_equal(owned[offs[i]: offs[i] + full[i].size],
                                   full[i].astype(np.float32).reshape(-1))
                    for i in full if owner[i] == rank)
    # the owner's "updates": a fresh seeded value per owned matrix element
    upd = {i: np.random.default_rng(100 + i).normal(size=full[i].shape).astype(np.float32)
           for i in full}
    for i in full:
        if owner[i] == rank:
            owned[offs[i]: offs[i] + full[i].size] = upd[i].reshape(-1)
    # step 5: owners -> shards (the same runs, reversed)
    back = torch.full((o["L"],), 7.0, dtype=torch.float32)
    ex.scatter_from_owners(dist, torch.from_numpy(owned), back)
    want = oref.scatter_updates(upd, o, [np.full(o["L"], 7.0) for _ in range(world)])[rank]
    ok_scatter = np.array_equal(back.numpy(), np.asarray(want, dtype=np.float32))
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{int(ok_gather)} {int(ok_scatter)} {len(ex.sends)} {len(ex.recvs)}\n")
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_gloo_ranks_exchange_to_owners_and_back(tmp_path, world):
    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mp.start_processes(_exchange_main, args=(world, port, str(tmp_path)), nprocs=world,
                       start_method="spawn")
    for r in range(world):
        g, sc, ns, nr = open(tmp_path / f"rank{r}.txt").read().split()
        assert g == "1" and sc == "1", (r, g, sc)
        assert int(ns) > 0
