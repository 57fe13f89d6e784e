"""A prefix state cache over a stack of Gated DeltaNet layers.

statecache.py (squad-0.8b, qev_fast, StateCache): a row [state prefix |
suffix] continues from the deepest cached state whose tokens it shares; the
state at chosen positions of the prefix is kept on the GPU, in an LRU bounded
in MB, for later rows. Per GDN layer a checkpoint is the fp32 recurrent state
and the last (kernel - 1) conv inputs before its position. Positions
(StateCache._bounds): every multiple of `stride`, p - `tail` and p itself,
each rounded down to `align` (64: the delta-rule chunk), where p is the
row's state length; no span between consecutive positions is longer than
the largest chunk (2048), extra positions being inserted to split longer
ones. A row restores the deepest checkpoint usable for it (_lookup: its
position is at most the longest common prefix with the row that made it) and
computes the rest; the checkpoints it makes form one group sharing that row's
prefix tokens; evicting a group's last checkpoint drops the group.

What runs where: the schedule, the lookup and the LRU are host bookkeeping
(this module); the restore is one gdn_state_copy launch over every layer
(pools flattened to [n_layers * slots]); the remaining tokens run through
gdn_prefill_chunked_ckpt per layer, which writes each new checkpoint's state
and conv tail straight into its cache slot from inside the chunked prefill.
The attention K/V, the router features and the slot routes the pages also
keep belong to other layer kinds and are not part of this path.
"""
from __future__ import annotations

from collections import OrderedDict

import numpy as np
import torch

from . import gdn

ACTS = ("q", "k", "v", "z", "a", "b")
WEIGHTS = ("A_log", "dt_bias", "conv_w", "norm_w")
LARGEST_CHUNK = 2048  # statecache.py CHUNKS[-1]


class _Group:
    """The checkpoints one row made, and the prefix tokens they share."""
    __slots__ = ("ids", "ckpts")

    def __init__(self, ids):
        self.ids = np.asarray(ids, dtype=np.int64)
        self.ckpts = []


class _Ckpt:
    __slots__ = ("group", "pos", "slot")

    def __init__(self, group, pos, slot):
        self.group, self.pos, self.slot = group, pos, slot


class PrefixSchedule:
    """The host bookkeeping of the cache (no GPU work): checkpoint positions,
    lookup, LRU eviction bounded in bytes, and the slot pool behind it.

    ckpt_bytes: device bytes one checkpoint holds (every layer's state and
    conv tail); mb: the budget in MiB; capacity = how many checkpoints fit."""

    def __init__(self, ckpt_bytes: int, mb: float, stride: int = 2048, tail: int = 16, align: int = 64,
                 largest_chunk: int = LARGEST_CHUNK):
        if align and stride % align:
            raise ValueError("stride must be a multiple of align (its multiples are checkpoint positions)")
        self.ckpt_bytes = int(ckpt_bytes)
        self.mb, self.stride, self.tail, self.align = mb, stride, tail, align
        self.largest_chunk = largest_chunk
        self.capacity = int(mb * 2**20) // self.ckpt_bytes
        self.ckpts: OrderedDict[int, _Ckpt] = OrderedDict()  # least recently used first
        self.groups: dict[int, _Group] = {}
        self.free = list(range(self.capacity - 1, -1, -1))  # slot stack, lowest slot on top
        self.stats = {"rows": 0, "hits": 0, "partial": 0, "cold": 0, "evicted": 0, "ckpts_made": 0,
                      "tokens_reused": 0, "tokens_computed": 0}

    @property
    def bytes(self) -> int:
        return len(self.ckpts) * self.ckpt_bytes

    def down(self, x: int) -> int:
        return x - x % self.align if self.align else x

    def bounds(self, c: int, p: int) -> list[int]:
        """Checkpoint positions of a state of p tokens computed from position c
        (StateCache._bounds): multiples of stride, p - tail and p, each rounded
        down to align, those above c, ascending, with extra positions so that
        no span is longer than the largest chunk."""
        e = self.down(p)
        b = {k for k in range(self.stride, e, self.stride) if k > c} if self.stride else set()
        if self.tail and self.down(p - self.tail) > c:
            b.add(self.down(p - self.tail))
        if e > c:
            b.add(e)
        out, s = [], c
        for x in sorted(b):
            while x - s > self.largest_chunk:
                s += self.largest_chunk
                out.append(s)
            out.append(x)
            s = x
        return out

    def lookup(self, x) -> list[_Ckpt]:
        """Checkpoints a row whose prefix tokens are x can use: each at a
        position no deeper than the prefix x shares with its group's row."""
        x = np.asarray(x, dtype=np.int64)
        out = []
        for g in self.groups.values():
            m = min(len(g.ids), len(x))
            if m == 0 or g.ids[0] != x[0]:
                continue
            ne = np.flatnonzero(g.ids[:m] != x[:m])
            lcp = int(ne[0]) if len(ne) else m
            out += [c for c in g.ckpts if c.pos <= lcp]
        return out

    def touch(self, c: _Ckpt):
        self.ckpts.move_to_end(id(c))

    def _evict_one(self):
        _, c = self.ckpts.popitem(last=False)
        c.group.ckpts.remove(c)
        if not c.group.ckpts:
            self.groups.pop(id(c.group), None)
        self.free.append(c.slot)
        self.stats["evicted"] += 1

    def allocate(self, n: int, keep=None) -> list[int]:
        """n free slots, evicting least recently used checkpoints as needed
        (never `keep`, the checkpoint a row is being restored from)."""
        if n > self.capacity - (1 if keep is not None else 0):
            raise ValueError(f"{n} checkpoints do not fit in a cache of {self.capacity}")
        if keep is not None and id(keep) in self.ckpts:
            self.touch(keep)
        while len(self.free) < n:
            if keep is not None and next(iter(self.ckpts)) == id(keep):
                self.ckpts.move_to_end(id(keep))
            self._evict_one()
        return [self.free.pop() for _ in range(n)]

    def plan(self, ids, state_len: int):
        """(checkpoint to restore or None, its position c0, the new checkpoint
        positions) for a row whose first state_len tokens are its state."""
        p = self.down(int(state_len))
        cands = self.lookup(np.asarray(ids[:p], dtype=np.int64)) if p > 0 else []
        best = max(cands, key=lambda c: c.pos) if cands else None
        c0 = best.pos if best is not None else 0
        return best, c0, (self.bounds(c0, int(state_len)) if c0 < p else [])

    def register(self, ids, state_len: int, positions, slots, best, c0: int, n: int):
        """Bookkeeping after a row: the new checkpoints (one group sharing the
        row's prefix), LRU order and statistics."""
        p = self.down(int(state_len))
        self.stats["rows"] += 1
        self.stats["hits" if c0 == p and p > 0 else ("partial" if c0 > 0 else "cold")] += 1
        self.stats["tokens_reused"] += c0
        self.stats["tokens_computed"] += n - c0
        if best is not None and id(best) in self.ckpts:
            self.touch(best)
        if positions:
            g = _Group(np.asarray(ids[:p], dtype=np.int64))
            self.groups[id(g)] = g
            for pos, slot in zip(positions, slots):
                ck = _Ckpt(g, pos, slot)
                g.ckpts.append(ck)
                self.ckpts[id(ck)] = ck
                self.stats["ckpts_made"] += 1


class PrefixStateCache:
    """The cache for a LayerStack: checkpoint slots on the device (fp32 states
    [n_layers][capacity][nv][dk][dv], bf16 conv tails [n_layers][capacity][3][C])
    behind a PrefixSchedule."""

    def __init__(self, stack, mb: float, stride: int = 2048, tail: int = 16, align: int = 64):
        if align % 64 != 0:
            raise ValueError("checkpoint positions must fall on chunk ends: align must be a multiple of 64")
        s = stack.shape
        self.stack = stack
        per = stack.n_layers * (s.nv * s.dk * s.dv * 4 + s.Kc * s.C * 2)
        self.sched = PrefixSchedule(per, mb, stride=stride, tail=tail, align=align)
        cap = max(1, self.sched.capacity)
        dev = stack.device
        self.ckpt_state = torch.zeros((stack.n_layers, cap, s.nv, s.dk, s.dv), dtype=torch.float32, device=dev)
        self.ckpt_conv = torch.zeros((stack.n_layers, cap, s.Kc, s.C), dtype=torch.bfloat16, device=dev)

    def _restore(self, best, slot: int):
        st, L = self.stack, self.stack.n_layers
        if best is None:  # a cold row starts from zeros (StateCache._restore(None))
            st.state_pool[:, slot].zero_()
            st.conv_pool[:, slot].zero_()
            return
        cap = self.ckpt_state.shape[1]
        src = torch.tensor([l * cap + best.slot for l in range(L)], dtype=torch.int32, device=st.device)
        dst = torch.tensor([l * st.n_slots + slot for l in range(L)], dtype=torch.int32, device=st.device)
        gdn.state_copy(st._dims(1, 1), self.ckpt_state, self.ckpt_conv, st.state_pool, st.conv_pool, src, dst, L,
                       L * cap, L * st.n_slots)

    def row(self, ids, state_len: int, acts, slot: int, out, workspace):
        """Run one row through every layer from the deepest usable checkpoint.

        ids: the row's tokens (n); acts[l][name]: layer l's inputs of the n
        tokens, [1, n, ...] on the device; slot: the row's slot in the stack's
        pools (its state on return is the state after all n tokens); out: bf16
        [n_layers][1][n][nv][dv], written for tokens c0 .. n-1. Returns c0, the
        tokens taken from the cache."""
        n = len(ids)
        sched = self.sched
        best, c0, positions = sched.plan(ids, state_len)
        slots = sched.allocate(len(positions), keep=best) if positions else []
        self._restore(best, slot)
        st = self.stack
        if n > c0:
            dims = st._dims(1, n - c0)
            idx = torch.tensor([slot], dtype=torch.int32, device=st.device)
            trip = (torch.tensor([[0, pos - c0, sl] for pos, sl in zip(positions, slots)], dtype=torch.int32,
                                 device=st.device) if positions else None)
            for l in range(st.n_layers):
                a = {k: acts[l][k][:, c0:n] for k in ACTS}
                w = st.weights[l]
                inp = gdn.make_inputs(*(a[k] for k in ACTS), *(w[k] for k in WEIGHTS), state_idx=idx)
                gdn.prefill_chunked_ckpt(dims, inp, st.conv_pool[l], st.state_pool[l], out[l][:, c0:n], workspace,
                                         trip, self.ckpt_state[l], self.ckpt_conv[l])
        sched.register(ids, state_len, positions, slots, best, c0, n)
        return c0
