"""A stack of Gated DeltaNet layers on per-layer state pools, stepped through the
C-ABI and captured in CUDA graphs.

uni_engine.py (Qwen3.5-9B-SpeedX9-GDN32): the decode runs as one captured CUDA
graph over every layer of the model, on cache tensors whose addresses never
change (copy_cache_ copies into them in place); statecache.py (squad-0.8b,
StateCache._graph / precapture): graphs are captured once per shape and
replayed with new inputs copied into their static buffers. generate.py
(sparkle, mlx_streaming/mtp): a speculative verify keeps each layer's state
after every draft token and commits the winning path's prefix.

Here a step of the stack is the layer calls of libgdn one after another (the
layers of this path are independent: no projection runs between them) plus,
for verify, one gdn_commit_accepted launch that commits every layer. The
pools are one tensor per kind, [n_layers][n_slots][...], so that a row keeps
one slot index in every layer (state_idx) and one launch reaches all layers.
The class only marshals buffers and issues the calls; the arithmetic is in
the library's kernels.
"""
from __future__ import annotations

import torch

from . import gdn

ACTS = ("q", "k", "v", "z", "a", "b")
WEIGHTS = ("A_log", "dt_bias", "conv_w", "norm_w")


def _act_shapes(shape, B, T):
    return {"q": (B, T, shape.kd), "k": (B, T, shape.kd), "v": (B, T, shape.vd), "z": (B, T, shape.vd),
            "a": (B, T, shape.nv), "b": (B, T, shape.nv)}


class LayerStack:
    """n_layers GDN layers sharing one head layout, with their recurrent-state
    and conv-tail pools of n_slots rows each.

    weights: one dict per layer with device tensors A_log, dt_bias, conv_w,
    norm_w. state_pool fp32 [n_layers][n_slots][nv][dk][dv] and conv_pool
    bf16 [n_layers][n_slots][3][C] are allocated here (zeros) and never
    reallocated."""

    def __init__(self, shape, weights, n_slots, device="cuda"):
        self.shape = shape
        self.n_layers = len(weights)
        self.n_slots = n_slots
        self.weights = weights
        self.device = device
        s = shape
        self.state_pool = torch.zeros((self.n_layers, n_slots, s.nv, s.dk, s.dv), dtype=torch.float32, device=device)
        self.conv_pool = torch.zeros((self.n_layers, n_slots, s.Kc, s.C), dtype=torch.bfloat16, device=device)

    def _dims(self, B, T):
        s = self.shape
        return gdn.make_dims(B=B, T=T, nk=s.nk, nv=s.nv, dk=s.dk, dv=s.dv, n_slots=self.n_slots)

    def _inputs(self, l, acts, state_idx):
        w = self.weights[l]
        return gdn.make_inputs(*(acts[n] for n in ACTS), *(w[n] for n in WEIGHTS), state_idx=state_idx)

    def static_acts(self, B, T):
        """Per-layer device buffers for a step of B rows x T tokens."""
        return [{n: torch.zeros(sh, dtype=torch.bfloat16, device=self.device)
                 for n, sh in _act_shapes(self.shape, B, T).items()} for _ in range(self.n_layers)]

    # ------------------------------------------------------------ eager steps

    def decode(self, acts, state_idx, out, stream=None):
        """One decode token for B rows through every layer: acts[l][name]
        [B,1,...], state_idx int32 [B] (device), out bf16 [n_layers][B][1][nv][dv]."""
        B = acts[0]["q"].shape[0]
        dims = self._dims(B, 1)
        for l in range(self.n_layers):
            gdn.decode_step(dims, self._inputs(l, acts[l], state_idx), self.conv_pool[l], self.state_pool[l], out[l],
                            stream)

    def verify(self, acts, state_idx, out, ckpt_state, ckpt_conv, stream=None):
        """Every layer's verify of B rows x T draft tokens from the pools (read
        only): out [n_layers][B][T][nv][dv], ckpt_state [n_layers][B][T][nv][dk][dv],
        ckpt_conv [n_layers][B][T][3][C]."""
        B, T = acts[0]["q"].shape[0], acts[0]["q"].shape[1]
        dims = self._dims(B, T)
        for l in range(self.n_layers):
            gdn.verify_with_checkpoints(dims, self._inputs(l, acts[l], state_idx), self.conv_pool[l],
                                        self.state_pool[l], out[l], ckpt_state[l], ckpt_conv[l], stream)

    def commit(self, paths, accept_len, dst_slot, ckpt_state, ckpt_conv, winner=None, stream=None):
        """Every layer's winning checkpoint into the pools, one launch."""
        B, T = ckpt_state.shape[1], ckpt_state.shape[2]
        gdn.commit_accepted(self._dims(B, T), self.n_layers, paths, ckpt_state, ckpt_conv, self.state_pool,
                            self.conv_pool, accept_len, dst_slot, winner, stream)

    # --------------------------------------------------------- captured steps

    def capture_decode(self, B):
        """A CUDA graph of one decode token for B rows through every layer.
        Copy a step's inputs into g.acts[l][name] and the rows' slots into
        g.state_idx, then g.replay(); outputs land in g.out."""
        return _Graph(self, "decode", B, 1)

    def capture_verify_commit(self, B, T, paths):
        """A CUDA graph of every layer's verify of B rows x T draft tokens
        followed by the fused commit of each group of `paths` rows. Before
        g.replay(): inputs into g.acts, slots into g.state_idx, accepted
        lengths into g.accept_len and each group's slot into g.dst_slot."""
        return _Graph(self, "verify_commit", B, T, paths)


class _Graph:
    def __init__(self, stack: LayerStack, kind, B, T, paths=1):
        s, dev = stack.shape, stack.device
        self.stack, self.kind, self.B, self.T, self.paths = stack, kind, B, T, paths
        self.acts = stack.static_acts(B, T)
        # rows of a decode step need distinct slots; verify rows may share one
        self.state_idx = (torch.arange(B, dtype=torch.int32, device=dev) % stack.n_slots if kind == "decode"
                          else torch.zeros(B, dtype=torch.int32, device=dev))
        self.out = torch.zeros((stack.n_layers, B, T, s.nv, s.dv), dtype=torch.bfloat16, device=dev)
        if kind == "verify_commit":
            self.ckpt_state = torch.zeros((stack.n_layers, B, T, s.nv, s.dk, s.dv), dtype=torch.float32, device=dev)
            self.ckpt_conv = torch.zeros((stack.n_layers, B, T, s.Kc, s.C), dtype=torch.bfloat16, device=dev)
            self.accept_len = torch.zeros(B, dtype=torch.int32, device=dev)
            self.dst_slot = torch.zeros(B // paths, dtype=torch.int32, device=dev)
            self.winner = torch.zeros(B // paths, dtype=torch.int32, device=dev)
        # one eager pass first (per-device first-use set-up happens outside the
        # capture), on a copy of the pools that is put back afterwards
        saved = (stack.state_pool.clone(), stack.conv_pool.clone())
        self._issue()
        torch.cuda.synchronize()
        stack.state_pool.copy_(saved[0])
        stack.conv_pool.copy_(saved[1])
        del saved
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._issue()
        torch.cuda.synchronize()

    def _issue(self):
        st = self.stack
        if self.kind == "decode":
            st.decode(self.acts, self.state_idx, self.out)
        else:
            st.verify(self.acts, self.state_idx, self.out, self.ckpt_state, self.ckpt_conv)
            st.commit(self.paths, self.accept_len, self.dst_slot, self.ckpt_state, self.ckpt_conv, self.winner)

    def replay(self):
        self.graph.replay()
