"""One Medusa draft-and-verify step as a sequence of C-ABI calls.

``MedusaStep`` owns the device buffers of one step for fixed shapes and
issues, in order: medusa_heads -> tree_attention (with the token fill) ->
lm_verify -> verify_accept -> compact_kv.  The tree is built once at
construction ("Medusa deep dive": the tree is chosen ahead of time).

Every buffer of the step is fixed at construction, so the whole step can be
recorded once as a CUDA graph (``capture``) and re-issued with a single
launch (``replay``): the step's dozen kernels then cost one host call.
"""
from __future__ import annotations

from typing import Dict, Optional, Sequence

import torch

from . import (BF16, F32, GREEDY, SAMPLE, TYPICAL, backbone_layer, backbone_workspace_size,
               build_tree_mask, compact_kv, dtype_code, embed_tokens, lm_verify,
               lm_verify_draft, lm_verify_sample, medusa_heads, mtp_heads, mtp_workspace_size,
               new_workspace, next_inputs, tree_attention, tree_size, verify_accept,
               verify_draft_workspace_size, workspace_size)


class MedusaStep:
    def __init__(self, *, W: torch.Tensor, lm: torch.Tensor, emb: torch.Tensor,
                 wqkv: torch.Tensor, wo: torch.Tensor, Kc: torch.Tensor, Vc: torch.Tensor,
                 P: torch.Tensor, shortlist: Sequence[int], max_rank_sum: int, Hq: int,
                 Hkv: int, B: int):
        dev = lm.device
        self.W, self.lm, self.emb, self.wqkv, self.wo = W, lm, emb, wqkv, wo
        self.Kc, self.Vc, self.P = Kc, Vc, P
        self.shortlist = tuple(int(s) for s in shortlist)
        self.max_rank_sum = int(max_rank_sum)
        self.K = len(self.shortlist)
        self.smax = max(self.shortlist)
        self.Hq, self.Hkv = Hq, Hkv
        self.B = B
        self.d = lm.shape[1]
        self.V = lm.shape[0]
        self.dh = Kc.shape[3]
        self.dtype = lm.dtype
        self.N = tree_size(self.shortlist, self.max_rank_sum)
        N, K, i32 = self.N, self.K, torch.int32
        words = (N + 63) // 64
        self.parent = torch.empty(N, dtype=i32, device=dev)
        self.depth = torch.empty(N, dtype=i32, device=dev)
        self.rank = torch.empty(N, dtype=i32, device=dev)
        self.mask = torch.empty((N, words), dtype=torch.int64, device=dev)
        build_tree_mask(self.shortlist, self.max_rank_sum, self.parent, self.depth, self.rank,
                        self.mask)
        self.U = torch.empty((B, K + 1, self.d), dtype=self.dtype, device=dev)
        self.root = torch.empty(B, dtype=i32, device=dev)
        # the heads' own argmax root in loop steps after the first, whose root
        # is the previous step's next_root
        self.root_draft = torch.empty(B, dtype=i32, device=dev)
        self._carried = False
        self.topk_id = torch.empty((B, K, self.smax), dtype=i32, device=dev)
        self.topk_val = torch.empty((B, K, self.smax), dtype=torch.float32, device=dev)
        self.tok = torch.empty((B, N), dtype=i32, device=dev)
        self.y = torch.empty((B, N, self.d), dtype=self.dtype, device=dev)
        self.argmax = torch.empty((B, N), dtype=i32, device=dev)
        self.stats = torch.empty((B, N, 4), dtype=torch.float32, device=dev)
        self.childlogit = torch.empty((B, N), dtype=torch.float32, device=dev)
        self.ok = torch.empty((B, N), dtype=torch.uint8, device=dev)
        self.L = torch.empty(B, dtype=i32, device=dev)
        self.path = torch.empty((B, K + 1), dtype=i32, device=dev)
        self.next_root = torch.empty(B, dtype=i32, device=dev)
        self.sample_id = torch.empty((B, N), dtype=i32, device=dev)
        nbytes = workspace_size(dtype_code(lm), B, self.d, self.V, K, N, Hq, Hkv, self.dh,
                                self.smax)
        # the fused verify pass (bf16): the next step's shortlists at every
        # tree row; its workspace need is added to the step's
        self.fused_ok = self.dtype == torch.bfloat16
        if self.fused_ok:
            self.tree_topk_id = torch.empty((B, N, K, self.smax), dtype=i32, device=dev)
            self.tree_topk_val = torch.empty((B, N, K, self.smax), dtype=torch.float32,
                                             device=dev)
            nbytes = max(nbytes, verify_draft_workspace_size(B, N, self.d, K))
        self.ws = new_workspace(nbytes, dev)

    def capture(self, h: torch.Tensor, mode: int = TYPICAL, eps: float = 0.09,
                delta: float = 0.3, commit: bool = True,
                h_host: Optional[torch.Tensor] = None, outputs_to_host: bool = False) -> None:
        """Record one step reading ``h`` into a CUDA graph.  Runs the step once
        eagerly first (on a side stream, so that every lazy set-up happens
        outside the capture); that run updates the KV cache and P like any
        step.  ``h`` must keep its storage: replays read it in place.

        ``h_host`` (pinned CPU tensor shaped like ``h``): every replay first
        copies it into ``h``.  ``outputs_to_host``: every replay ends by
        copying L, path, the tree tokens and next_root into pinned CPU
        tensors, available as ``self.host_out`` once the replay's stream has
        been synchronised.  A step then costs one graph launch."""
        dev = h.device
        if h_host is not None and (h_host.is_cuda or not h_host.is_pinned()):
            raise ValueError("h_host must be a pinned CPU tensor")
        self.host_out = None
        if outputs_to_host:
            self.host_out = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory()
                             for k, v in (("L", self.L), ("path", self.path), ("tok", self.tok),
                                          ("next_root", self.next_root))}

        def body():
            if h_host is not None:
                h.copy_(h_host, non_blocking=True)
            self.run(h, mode, eps, delta, commit)
            if self.host_out is not None:
                for k, src in (("L", self.L), ("path", self.path), ("tok", self.tok),
                               ("next_root", self.next_root)):
                    self.host_out[k].copy_(src, non_blocking=True)

        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            body()
        torch.cuda.current_stream(dev).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            body()
        self._graph = graph

    def replay(self) -> None:
        """Enqueue the captured step on the current stream (asynchronous)."""
        if getattr(self, "_graph", None) is None:
            raise RuntimeError("capture() has not been called")
        self._graph.replay()

    def run(self, h: torch.Tensor, mode: int = TYPICAL, eps: float = 0.09,
            delta: float = 0.3, commit: bool = True, temperature: float = 1.0,
            seed: int = 0) -> None:
        """Enqueue one step on the current stream (asynchronous).  mode GREEDY,
        TYPICAL or SAMPLE (exact sampling at ``temperature`` with key
        ``seed``).  A single step: its root is the base head's argmax, and a
        decoding loop started after it begins afresh."""
        self._carried = False
        self._draft(h)
        self._verify_layers()
        self._verify_and_accept(mode, eps, delta, temperature, seed)
        if commit:
            self._commit()

    def _draft(self, h, root=None):
        """The step's draft from hidden state h: U, root (into ``root`` when
        given, else self.root) and shortlists."""
        medusa_heads(h, self.W, self.lm, self.shortlist, self.smax, self.U,
                     self.root if root is None else root, self.topk_id, self.topk_val, self.ws)

    def _before_commit(self):
        pass

    def _next(self, h, fused):
        """The next step's inputs (after the commit)."""
        if fused:
            next_inputs(self.L, self.path, self.ws, N=self.N, smax=self.smax,
                        next_root=self.next_root, y=self.y, tree_topk_id=self.tree_topk_id,
                        tree_topk_val=self.tree_topk_val, h_next=h, root_out=self.root,
                        topk_id_out=self.topk_id, topk_val_out=self.topk_val)
        else:
            next_inputs(self.L, self.path, self.ws, N=self.N, smax=self.smax,
                        next_root=self.next_root, y=self.y, h_next=h, root_out=self.root)

    def _verify_layers(self):
        """Token fill and the verify layer(s): y for every tree row."""
        tree_attention(self.P, self.tok, self.mask, self.emb, self.wqkv, self.wo, self.Kc,
                       self.Vc, self.y, self.ws, Hq=self.Hq, Hkv=self.Hkv, K=self.K,
                       smax=self.smax, root=self.root, topk_id=self.topk_id, depth=self.depth,
                       rank=self.rank)

    def _commit(self):
        """Commit the accepted path's KV and advance P."""
        compact_kv(self.L, self.path, self.Kc, self.Vc, self.P, self.ws)

    def _verify_and_accept(self, mode, eps, delta, temperature, seed, fused=False):
        if fused:
            if mode == SAMPLE:
                raise ValueError("exact sampling runs with the separate verify pass")
            lm_verify_draft(self.y, self.W, self.lm, self.shortlist, self.smax, self.tok,
                            self.parent, self.argmax, self.stats, self.childlogit,
                            self.tree_topk_id, self.tree_topk_val, self.ws)
        elif mode == SAMPLE:
            lm_verify_sample(self.y, self.lm, self.tok, self.parent, self.P, temperature, seed,
                             self.argmax, self.stats, self.childlogit, self.sample_id, self.ws)
        else:
            lm_verify(self.y, self.lm, self.tok, self.parent, self.argmax, self.stats,
                      self.childlogit, self.ws)
        verify_accept(mode, eps, delta, self.parent, self.depth, self.tok,
                      self.sample_id if mode == SAMPLE else self.argmax, self.stats,
                      self.childlogit, self.L, self.path, self.next_root, self.ws, ok=self.ok)

    # ------------------------------------------------------------------
    # The decoding loop ("Medusa Heads", "How it works": draft, verify,
    # accept and roll back, then draft again from the last accepted
    # position).  Step s + 1 reads the verify layer's output at step s's
    # accepted node as its hidden state; its root is step s's next_root (the
    # token the base model supplies after the accepted prefix: the argmax at
    # the accepted node under greedy and typical acceptance, the token drawn
    # there under exact sampling).
    #
    # Two forms of the steady-state step:
    #   separate (canonical order): medusa_heads(h) -> tree_attention ->
    #       lm_verify -> verify_accept -> compact_kv -> next_inputs(root, h)
    #       (two LM-projection streams per step: draft rows, verify rows);
    #   fused: tree_attention -> lm_verify_draft -> verify_accept ->
    #       compact_kv -> next_inputs(root, shortlists, h): the K heads run on
    #       every tree row and one LM-projection stream serves the verify
    #       rows and the next step's draft rows.  The first step of a loop
    #       drafts with medusa_heads.
    # The fused form trades a second weight stream for (K + 1) times the
    # verify rows in one pass; it pays only while those rows keep the pass
    # at its weight-stream time.  Measured on the Vicuna-7B-shaped batch-1
    # workload (89 tree rows, 445 rows in the fused pass): 363 us per fused
    # step against 247 us separate, so "auto" keeps the separate form above
    # one 128-row tile (``FUSED_MAX_ROWS``).
    # ------------------------------------------------------------------

    # Largest B N (K + 1) for which "auto" picks the fused form.
    FUSED_MAX_ROWS = 128

    def fused_auto(self) -> bool:
        return (self.fused_ok and self.W is not None
                and self.B * self.N * (self.K + 1) <= self.FUSED_MAX_ROWS)

    def begin_decode(self, h: torch.Tensor, fused: bool, root: torch.Tensor = None) -> None:
        """Before the first step of a loop: the fused form drafts the first
        step from ``h`` (root and shortlists); the separate form drafts in
        its first step.  The first root is the base head's argmax unless
        ``root`` (device [B] int32) gives it, e.g. the prefill's own draw
        under exact sampling."""
        self._carried = False
        if fused:
            if not self.fused_ok:
                raise ValueError("the fused verify pass needs bf16 weights")
            self._draft(h)
        if root is not None:
            self.root.copy_(root)
            self._carried = True

    def decode_step(self, h: torch.Tensor, fused: bool, mode: int = TYPICAL, eps: float = 0.09,
                    delta: float = 0.3, temperature: float = 1.0, seed: int = 0) -> None:
        """Enqueue one steady-state step (asynchronous).  Updates in place:
        the KV caches and P (the accepted path committed), ``h`` (the next
        step's hidden state) and, in the fused form, root / topk_id /
        topk_val (the next step's draft) or root alone (the separate form,
        whose next step drafts its shortlists from ``h``)."""
        if not fused:
            # after the first step the root is already in place (the last
            # step's next_root); the heads' own argmax is not used
            self._draft(h, self.root_draft if self._carried else None)
        self._verify_layers()
        self._verify_and_accept(mode, eps, delta, temperature, seed, fused)
        self._before_commit()
        self._commit()
        self._next(h, fused)
        self._carried = True

    def decode(self, h: torch.Tensor, n_steps: int, fused="auto", mode: int = TYPICAL,
               eps: float = 0.09, delta: float = 0.3, record: bool = False,
               temperature: float = 1.0, seed: int = 0, root: torch.Tensor = None):
        """``n_steps`` consecutive steps from hidden state ``h`` (updated in
        place).  ``fused``: True, False or "auto" (``fused_auto``).  ``root``:
        the first step's root (see ``begin_decode``).  With ``record`` the
        host waits after every step and the per-step L, path, tree tokens and
        next_root are returned (host tensors)."""
        if fused == "auto":
            fused = self.fused_auto() and mode != SAMPLE
        self.begin_decode(h, fused, root)
        out = []
        for _ in range(n_steps):
            self.decode_step(h, fused, mode, eps, delta, temperature, seed)
            if record:
                torch.cuda.current_stream(h.device).synchronize()
                out.append(dict(L=self.L.cpu(), path=self.path.cpu(), tok=self.tok.cpu(),
                                next_root=self.next_root.cpu()))
        return out


class BackboneStep(MedusaStep):
    """A Medusa step whose verify pass is a backbone of several layers with
    the tree's position ids ("Medusa deep dive", "From top-k heads to a
    sparse candidate tree": the tree is a flat node sequence with an attention
    mask and position ids, pushed through the backbone in one pass).

    ``layers``: one dict per layer with ``wqkv`` [(Hq + 2 Hkv) dh, d], ``wo``
    [d, Hq dh], ``Kc``, ``Vc`` [B, Hkv, Pmax, dh] (each layer's own cache).
    x_0 = Emb[tok]; layer l: q, k rotated to P_b + depth_n, attention, and
    x_l = x_{l-1} + Wo_l o_l; the verify logits read x_L.  Every layer's
    cache gets the accepted path committed.  bf16 only."""

    def __init__(self, *, layers, rope_base: float = 10000.0, **kw):
        l0 = layers[0]
        super().__init__(wqkv=l0["wqkv"], wo=l0["wo"], Kc=l0["Kc"], Vc=l0["Vc"], **kw)
        if self.dtype != torch.bfloat16:
            raise ValueError("the backbone form of the verify pass is bf16 only")
        self.layers = list(layers)
        self.rope_base = float(rope_base)
        dev = self.lm.device
        shape = (self.B, self.N, self.d)
        self.xbuf = [torch.empty(shape, dtype=self.dtype, device=dev) for _ in range(2)]
        self.P_scratch = torch.empty_like(self.P)
        need = backbone_workspace_size(self.B, self.N, self.d, self.Hq, self.Hkv, self.dh)
        if need > self.ws.numel():
            self.ws = new_workspace(need, dev)

    def _verify_layers(self):
        embed_tokens(self.tok, self.emb, self.xbuf[0], self.ws, K=self.K, smax=self.smax,
                     root=self.root, topk_id=self.topk_id, depth=self.depth, rank=self.rank)
        L = len(self.layers)
        for l, lw in enumerate(self.layers):
            src = self.xbuf[l % 2]
            dst = self.y if l == L - 1 else self.xbuf[(l + 1) % 2]
            backbone_layer(self.P, self.depth, self.mask, src, lw["wqkv"], lw["wo"], lw["Kc"],
                           lw["Vc"], dst, self.ws, Hq=self.Hq, Hkv=self.Hkv,
                           rope_base=self.rope_base)

    def _commit(self):
        # every layer's cache takes the path at the same P; P advances once
        for lw in self.layers[:-1]:
            self.P_scratch.copy_(self.P)
            compact_kv(self.L, self.path, lw["Kc"], lw["Vc"], self.P_scratch, self.ws)
        last = self.layers[-1]
        compact_kv(self.L, self.path, last["Kc"], last["Vc"], self.P, self.ws)


class MTPStep(MedusaStep):
    """A Medusa step drafted by MTP-style heads ("Speculative Decoding Deep
    Dive II: Medusa, MTP", section "MTP": n heads on h_t that are transformer
    layers, one shared unembedding, used with Medusa's tree and verification).

    ``heads``: K dicts with ``wqkv``, ``wo`` (attention, as a backbone layer),
    ``w1`` [dff, d], ``w2`` [d, dff] (the MLP) and ``Kc``, ``Vc`` (the head's
    own cache).  Each draft hands the heads the hidden states of the last
    step's accepted tokens (h alone, at position P_b - 1, for the first step
    of a loop).  The separate form of the loop only (the fused verify pass
    drafts with residual-block heads)."""

    def __init__(self, *, heads, rope_base: float = 10000.0, **kw):
        kw.setdefault("W", None)
        super().__init__(**kw)
        if self.dtype != torch.bfloat16:
            raise ValueError("MTP heads are bf16 only")
        if len(heads) != self.K:
            raise ValueError("one MTP head per shortlist entry")
        self.heads = list(heads)
        self.rope_base = float(rope_base)
        dev = self.lm.device
        K, i32 = self.K, torch.int32
        chain = (1,) * K
        self.chain_parent = torch.empty(K + 1, dtype=i32, device=dev)
        self.chain_depth = torch.empty(K + 1, dtype=i32, device=dev)
        self.chain_rank = torch.empty(K + 1, dtype=i32, device=dev)
        self.chain_mask = torch.empty((K + 1, 1), dtype=torch.int64, device=dev)
        build_tree_mask(chain, -1, self.chain_parent, self.chain_depth, self.chain_rank,
                        self.chain_mask)
        self.xrows = torch.empty((self.B, K + 1, self.d), dtype=self.dtype, device=dev)
        self.Lm = torch.zeros(self.B, dtype=i32, device=dev)
        self.P0 = torch.empty_like(self.P)
        dff = heads[0]["w1"].shape[0]
        need = mtp_workspace_size(self.B, K, self.d, dff, self.Hq, self.Hkv, self.dh)
        if need > self.ws.numel():
            self.ws = new_workspace(need, dev)
        self.fused_ok = False

    def _start(self, h):
        """The heads' rows from h alone: row 0 = h at position P_b - 1, the
        others padding (copies of h)."""
        self.xrows.copy_(h[:, None, :].expand_as(self.xrows))
        self.Lm.zero_()
        torch.sub(self.P, 1, out=self.P0)

    def run(self, h, *args, **kw):
        self._start(h)
        super().run(h, *args, **kw)

    def begin_decode(self, h, fused, root=None):
        if fused:
            raise ValueError("MTP heads run with the separate form of the loop")
        self._carried = False
        self._start(h)
        if root is not None:
            self.root.copy_(root)
            self._carried = True

    def _draft(self, h, root=None):
        mtp_heads(self.xrows, self.Lm, self.P0, self.chain_depth, self.chain_mask, self.heads,
                  self.lm, self.shortlist, self.smax, self.U,
                  self.root if root is None else root, self.topk_id, self.topk_val, self.ws,
                  Hq=self.Hq, Hkv=self.Hkv, rope_base=self.rope_base)

    def _before_commit(self):
        self.P0.copy_(self.P)            # position of the accepted rows' first

    def _next(self, h, fused):
        next_inputs(self.L, self.path, self.ws, N=self.N, smax=self.smax,
                    next_root=self.next_root, y=self.y, h_next=h, root_out=self.root,
                    rows_out=self.xrows)
        self.Lm.copy_(self.L)
