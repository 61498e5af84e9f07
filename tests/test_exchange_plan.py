"""The owner exchange plan ("Add initial Muon+M-FSDPv2 implementation", "Opt step" steps 3
and 5): per rank, the runs of matrix elements sent to owners and received from shard
holders.  Host only: the library's planner is checked by brute force on tiny layouts, and
moving the data with torch.distributed on CPU tensors (gloo, 2 and 3 ranks) rebuilds, bit
for bit, what the oracle's gather gives on each owner and, on the way back, what its
scatter gives on each shard."""
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
    from oracle import muon_ref as oref
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # straddling parameters: the ragged set plus a vector, split over `world` shards
    wl = inp.WORKLOADS["ragged_small"]
    shapes = list(wl.shapes) + [(1000, 1), (97, 113)]
    flags = list(wl.is_matrix) + [False, True]
    lay = c.muon_layout_create(shapes, world, 0, flags)
    owner, _ = c.muon_assign_owners(lay)
    sends, recvs, owned_numel, offs = c.muon_exchange_plan(lay, owner, rank)
    o = oref.flat_layout(shapes, world, flags)
    flat = np.random.default_rng(11).normal(size=lay.numel).astype(np.float32)
    my_shard = oref.shard_flat(flat, o)[rank].astype(np.float32)

    def move(src_lists, dst_lists, read, write):
        """One message per peer: the runs to that peer back to back, in list order."""
        reqs = []
        for peer in range(world):
            out = [x for x in src_lists if x["dst_rank" if read == "shard" else "src_rank"] == peer]
            if not out:
                continue
            buf = np.concatenate([read_run(x, read) for x in out]).astype(np.float32)
            if peer == rank:
                local[peer] = buf
            else:
                reqs.append(dist.isend(torch.from_numpy(buf), dst=peer))
        for peer in range(world):
            inc = [x for x in dst_lists if x["src_rank" if read == "shard" else "dst_rank"] == peer]
            if not inc:
                continue
            n = sum(x["len"] for x in inc)
            if peer == rank:
                buf = local[peer]
            else:
                t = torch.empty(n, dtype=torch.float32)
                dist.recv(t, src=peer)
                buf = t.numpy()
            pos = 0
            for x in inc:
                write_run(x, write, buf[pos: pos + x["len"]])
                pos += x["len"]
        for q in reqs:
            q.wait()

    owner_buf = np.full(max(1, owned_numel), np.nan, dtype=np.float32)
    shard_back = np.full(o["L"], 7.0, dtype=np.float32)

    def read_run(x, where):
        if where == "shard":
            return my_shard[x["shard_off"]: x["shard_off"] + x["len"]]
        return owner_buf[x["owner_off"]: x["owner_off"] + x["len"]]

    def write_run(x, where, vals):
        if where == "owner":
            owner_buf[x["owner_off"]: x["owner_off"] + x["len"]] = vals
        else:
            shard_back[x["shard_off"]: x["shard_off"] + x["len"]] = vals

    local = {}
    # step 3: shards -> owners
    move(sends, recvs, "shard", "owner")
    full = oref.gather_full(oref.shard_flat(flat, o), o)
    ok_gather = all(np.array_equal(owner_buf[offs[i]: offs[i] + full[i].size],
                                   full[i].astype(np.float32).reshape(-1))
                    for i in full if owner[i] == rank)
    # the owner's "updates": a fresh seeded value per owned matrix element
    upd = {i: np.random.default_rng(100 + i).normal(size=full[i].shape).astype(np.float32)
           for i in full}
    for i in full:
        if owner[i] == rank:
            owner_buf[offs[i]: offs[i] + full[i].size] = upd[i].reshape(-1)
    # step 5: owners -> shards (the same runs, reversed)
    local = {}
    move(recvs, sends, "owner", "shard")
    want = oref.scatter_updates(upd, o, [np.full(o["L"], 7.0) for _ in range(world)])[rank]
    ok_scatter = np.array_equal(shard_back, np.asarray(want, dtype=np.float32))
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{int(ok_gather)} {int(ok_scatter)} {len(sends)} {len(recvs)}\n")
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
