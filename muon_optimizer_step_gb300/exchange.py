"""Owner exchange over torch.distributed: move the runs muon_exchange_plan lists.

"Add initial Muon+M-FSDPv2 implementation", "Opt step" step 3: each sharded matrix's
orthogonalization input is gathered on its owner; step 5: the owner's update is sent back
to the ranks that hold the matrix's shards.  The plan (which runs go where, and where they
land in the owner's packed buffer) comes from the library's host planner; this module only
packs each peer's runs into one message, sends and receives them with torch.distributed
point-to-point calls, and unpacks them.  It works on whichever backend the process group
uses (gloo with CPU tensors, NCCL with CUDA tensors).

With one GPU per process, the optimizer step itself emulates the owner as indexing (the
gather and scatter fused into its kernels); this module is the data plane for a real
multi-rank group.
"""
from __future__ import annotations

from . import capi


class OwnerExchange:
    """The exchange plan of one rank: runs sent to owners and received from shard holders.

    layout: a capi.Layout with one shard per rank; owner: one owner rank per parameter
    (capi.muon_assign_owners gives one); rank: this process's rank.
    """

    def __init__(self, layout, owner, rank):
        self.layout = layout
        self.rank = int(rank)
        self.owner = list(owner)
        self.sends, self.recvs, self.owned_numel, self.owned_offsets = \
            capi.muon_exchange_plan(layout, owner, rank)

    def _by_peer(self, runs, key):
        out = {}
        for x in runs:
            out.setdefault(x[key], []).append(x)
        return out

    def _move(self, dist, out_runs, out_key, read, in_runs, in_key, write, dtype, device, group):
        """One message per peer: the runs for that peer back to back, in list order.  All
        sends and receives are posted together (batch_isend_irecv), then unpacked."""
        import torch
        ops, local, inbox = [], None, []
        for peer, runs in sorted(self._by_peer(out_runs, out_key).items()):
            msg = torch.cat([read(x) for x in runs]).contiguous()
            if peer == self.rank:
                local = msg
            else:
                ops.append(dist.P2POp(dist.isend, msg, peer, group))
        for peer, runs in sorted(self._by_peer(in_runs, in_key).items()):
            if peer == self.rank:
                inbox.append((runs, None))
            else:
                msg = torch.empty(sum(x["len"] for x in runs), dtype=dtype, device=device)
                ops.append(dist.P2POp(dist.irecv, msg, peer, group))
                inbox.append((runs, msg))
        if ops:
            for q in dist.batch_isend_irecv(ops):
                q.wait()
        for runs, msg in inbox:
            msg = local if msg is None else msg
            pos = 0
            for x in runs:
                write(x, msg[pos: pos + x["len"]])
                pos += x["len"]

    def gather_to_owners(self, dist, shard, group=None):
        """Step 3: this rank's shard (a 1-D tensor of the layout's shard length) in, this
        rank's packed owner buffer out: every matrix it owns, row-major, at
        owned_offsets[i]."""
        import torch
        buf = torch.zeros(max(1, self.owned_numel), dtype=shard.dtype, device=shard.device)

        def read(x):
            return shard[x["shard_off"]: x["shard_off"] + x["len"]]

        def write(x, vals):
            buf[x["owner_off"]: x["owner_off"] + x["len"]] = vals
        self._move(dist, self.sends, "dst_rank", read, self.recvs, "src_rank", write,
                   shard.dtype, shard.device, group)
        return buf

    def scatter_from_owners(self, dist, owned, shard, group=None):
        """Step 5: this rank's packed owner buffer in; every run of its shard that belongs
        to a matrix is overwritten with the owner's values (other positions untouched)."""
        def read(x):
            return owned[x["owner_off"]: x["owner_off"] + x["len"]]

        def write(x, vals):
            shard[x["shard_off"]: x["shard_off"] + x["len"]] = vals
        self._move(dist, self.recvs, "src_rank", read, self.sends, "dst_rank", write,
                   shard.dtype, shard.device, group)
        return shard
