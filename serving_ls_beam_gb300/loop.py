"""Device-resident autoregressive beam-search loop over the C ABI.

One decode step is ``ls_beam_step`` (select the k best (token, parent) pairs of
every batch from that step's logits) followed by ``ls_cache_reorder`` (gather
the KV cache rows by parent beam, positions [0, t)), with the step's scores and
finished flags becoming the next step's beam state.  Everything stays on the
GPU: the beam state and the two cache buffers alternate between two sets
(ping-pong), so a run of steps can be captured in one CUDA graph.

With ``inplace=True`` the cache is one buffer refreshed in place, copy on change
(``ls_cache_refresh_inplace``): rows that continue themselves are not moved.

``step_projection`` takes the decoder states and the output projection instead of logits
(``ls_logits_beam_step``: the logits are made on the tensor cores and never stored).

With ``max_steps`` > 0 every step writes its tokens and parents straight into a
[max_steps, batch, k] history, and ``finalize`` turns the history into the token
sequence and length of every final beam (``ls_backtrack``): the n-best list of each
batch, best first, for a search stopped at the length limit or when every beam finished.

Follows the LightSeq inference article (31duo.com, itemid-283120): decoding =
vocab softmax + beam selection + cache refresh per step, with every buffer
allocated once at its static maximum (memory-reuse section).
"""
from __future__ import annotations

import torch

from . import (check, ls_backtrack, ls_beam_step, ls_beam_step_workspace_size, ls_cache_refresh_inplace,
               ls_cache_reorder, ls_logits_beam_step, ls_workspace_init)


class BeamSearchLoop:
    def __init__(self, batch: int, k: int, vocab: int, eos_id: int, kv_shape=None, kv_dtype=torch.float16,
                 device="cuda", caches=None, max_steps: int = 0, inplace: bool = False):
        """kv_shape = (layers, heads, max_len, head_dim) or None for no cache refresh.
        caches: optional pair of preallocated [layers, batch*k, heads, max_len, head_dim] tensors.
        max_steps: length limit of a search; > 0 keeps the token / parent history for finalize().
        inplace: refresh one cache buffer in place (caches[0] when given) instead of ping-pong."""
        self.batch, self.k, self.vocab, self.eos_id = batch, k, vocab, eos_id
        self.device = torch.device(device)
        dev = self.device
        self.workspace = torch.empty(ls_beam_step_workspace_size(batch, k, vocab), dtype=torch.uint8, device=dev)
        check(ls_workspace_init(self.workspace), "ls_workspace_init")
        # two sets of beam state: set s is read by a step, set 1-s written by it
        self.scores = [torch.zeros(batch, k, dtype=torch.float32, device=dev) for _ in range(2)]
        self.finished = [torch.zeros(batch, k, dtype=torch.uint8, device=dev) for _ in range(2)]
        self.token = [torch.zeros(batch, k, dtype=torch.int32, device=dev) for _ in range(2)]
        self.parent = [torch.zeros(batch, k, dtype=torch.int32, device=dev) for _ in range(2)]
        self.kv_shape = kv_shape
        if kv_shape is not None:
            layers, heads, max_len, head_dim = kv_shape
            shape = (layers, batch * k, heads, max_len, head_dim)
            if caches is None:
                caches = [torch.zeros(shape, dtype=kv_dtype, device=dev) for _ in range(1 if inplace else 2)]
            self.cache = list(caches)[:1] if inplace else list(caches)
        else:
            self.cache = None
        self.cur = 0
        self.inplace = inplace
        self.max_steps = max_steps
        if max_steps > 0:
            self.token_hist = torch.zeros(max_steps, batch, k, dtype=torch.int32, device=dev)
            self.parent_hist = torch.zeros(max_steps, batch, k, dtype=torch.int32, device=dev)
            self.seq_buf = torch.empty(batch * k * max_steps, dtype=torch.int32, device=dev)
            self.seq_len = torch.empty(batch, k, dtype=torch.int32, device=dev)
        self._last = (self.token[0], self.parent[0])

    def token_out(self, t: int) -> torch.Tensor:
        """Where decode step t (1-based) writes its tokens: the history slice, or the next state set."""
        return self.token_hist[t - 1] if self.max_steps > 0 else self.token[1 - self.cur]

    def parent_out(self, t: int) -> torch.Tensor:
        return self.parent_hist[t - 1] if self.max_steps > 0 else self.parent[1 - self.cur]

    def reset(self, beam_scores=None, finished=None):
        """Start a new search: beam state set 0 from the given tensors (default: scores 0, none finished)."""
        self.cur = 0
        if beam_scores is None:
            self.scores[0].zero_()
        else:
            self.scores[0].copy_(beam_scores)
        if finished is None:
            self.finished[0].zero_()
        else:
            self.finished[0].copy_(finished)

    def step(self, logits: torch.Tensor, t: int, bias=None, stream=None) -> int:
        """Decode step t (1-based): beam step on `logits` [batch, k, vocab], then the cache refresh of
        positions [0, t).  Returns the index of the state set holding this step's outputs."""
        return self._advance(t, stream, lambda s, n, tok, par: check(
            ls_beam_step(logits, bias, self.scores[s], self.finished[s], self.eos_id, tok, par, self.scores[n],
                         self.finished[n], self.workspace, stream), "ls_beam_step"))

    def step_projection(self, hidden: torch.Tensor, weight: torch.Tensor, t: int, bias=None, stream=None) -> int:
        """Decode step t (1-based) from the decoder states `hidden` [batch, k, dim] and the output projection
        `weight` [vocab, dim] (f16 or bf16; logits = hidden . weight^T, never stored), then the cache refresh
        of positions [0, t).  Returns the index of the state set holding this step's outputs."""
        return self._advance(t, stream, lambda s, n, tok, par: check(
            ls_logits_beam_step(hidden, weight, bias, self.scores[s], self.finished[s], self.eos_id, tok, par,
                                self.scores[n], self.finished[n], self.workspace, stream), "ls_logits_beam_step"))

    def _advance(self, t: int, stream, beam_step) -> int:
        if self.max_steps > 0 and not 1 <= t <= self.max_steps:
            raise ValueError(f"decode step {t} outside 1..{self.max_steps}")
        s, n = self.cur, 1 - self.cur
        tok, par = self.token_out(t), self.parent_out(t)
        beam_step(s, n, tok, par)
        if self.cache is not None:
            if self.inplace:
                check(ls_cache_refresh_inplace(self.cache[0], par, t, self.workspace, stream),
                      "ls_cache_refresh_inplace")
            else:
                check(ls_cache_reorder(self.cache[s], self.cache[n], par, t, stream=stream), "ls_cache_reorder")
        self.cur = n
        self._last = (tok, par)
        return n

    def current_cache(self):
        """The cache buffer holding the latest step's refresh."""
        return self.cache[0] if self.inplace else self.cache[self.cur]

    def outputs(self, idx: int | None = None):
        """The last step's tokens and parents with the beam state of set idx (default: the current one)."""
        i = self.cur if idx is None else idx
        return {"token": self._last[0], "parent": self._last[1], "score": self.scores[i],
                "finished": self.finished[i]}

    def finalize(self, steps: int, stream=None):
        """Token sequences [batch, k, steps] and lengths [batch, k] of the final beams after `steps` decode
        steps (best beam first), read back through the parent history on the device."""
        if self.max_steps <= 0:
            raise ValueError("the loop keeps no history (max_steps = 0)")
        if not 1 <= steps <= self.max_steps:
            raise ValueError(f"steps {steps} outside 1..{self.max_steps}")
        seq = self.seq_buf[: self.batch * self.k * steps].view(self.batch, self.k, steps)
        check(ls_backtrack(self.token_hist[:steps], self.parent_hist[:steps], self.eos_id, seq, self.seq_len,
                           self.workspace, stream), "ls_backtrack")
        return seq, self.seq_len
