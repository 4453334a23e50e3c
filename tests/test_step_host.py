"""Host logic of the decoding loop in MedusaStep, on the CPU: which root each
step's tree is filled from.  The calls that launch kernels are replaced by
recorders (a fake draft root of 7 from the heads, next_root = 100 + step);
the loop's own code runs unchanged."""
from __future__ import annotations

import pytest
import torch

import speculative_decoding_08_b300 as mds
from speculative_decoding_08_b300 import step as st

B, D, V, HQ, HKV, DH, PMAX = 2, 64, 50, 2, 1, 64, 64
SHORTLIST = (2, 2)


@pytest.fixture
def fake(monkeypatch):
    log = {"tree_root": [], "heads_root": [], "steps": 0}

    def build_tree_mask(shortlist, max_rank_sum, parent, depth, rank, mask):
        return parent.numel()

    def medusa_heads(h, W, lm, shortlist, smax, U, root, topk_id, topk_val, ws):
        root.fill_(7)
        log["heads_root"].append(root)

    def tree_attention(P, tok, mask, emb, wqkv, wo, Kc, Vc, y, ws, **kw):
        tok[:, 0] = kw["root"]
        log["tree_root"].append(kw["root"].tolist())

    def verify_accept(mode, eps, delta, parent, depth, tok, argmax, stats, child, L, path,
                      next_root, ws, ok=None):
        next_root.fill_(100 + log["steps"])
        L.zero_()
        path.zero_()
        log["steps"] += 1

    def next_inputs(L, path, ws, *, N, smax, next_root=None, root_out=None, **kw):
        if root_out is not None:
            root_out.copy_(next_root)

    def nothing(*args, **kw):
        pass

    for name, fn in (("build_tree_mask", build_tree_mask), ("medusa_heads", medusa_heads),
                     ("tree_attention", tree_attention), ("verify_accept", verify_accept),
                     ("next_inputs", next_inputs), ("lm_verify", nothing),
                     ("lm_verify_sample", nothing), ("compact_kv", nothing)):
        monkeypatch.setattr(st, name, fn)
    return log


def make_step():
    z = torch.zeros
    return st.MedusaStep(W=z(len(SHORTLIST), D, D), lm=z(V, D), emb=z(V, D),
                         wqkv=z((HQ + 2 * HKV) * DH, D), wo=z(D, HQ * DH),
                         Kc=z(B, HKV, PMAX, DH), Vc=z(B, HKV, PMAX, DH),
                         P=torch.full((B,), 5, dtype=torch.int32), shortlist=SHORTLIST,
                         max_rank_sum=-1, Hq=HQ, Hkv=HKV, B=B)


def test_separate_loop_roots_follow_next_root(fake):
    """First step: the heads' argmax; later steps: the last step's next_root,
    the heads' own argmax going to scratch."""
    s = make_step()
    h = torch.zeros(B, D)
    s.begin_decode(h, False)
    for _ in range(3):
        s.decode_step(h, False, mds.SAMPLE, 0.0, 0.0, 1.0, 0)
    assert fake["tree_root"] == [[7, 7], [100, 100], [101, 101]]
    assert fake["heads_root"][0] is s.root
    assert all(r is s.root_draft for r in fake["heads_root"][1:])


def test_given_first_root(fake):
    s = make_step()
    h = torch.zeros(B, D)
    s.begin_decode(h, False, torch.tensor([42, 43], dtype=torch.int32))
    for _ in range(2):
        s.decode_step(h, False, mds.SAMPLE, 0.0, 0.0, 1.0, 0)
    assert fake["tree_root"] == [[42, 43], [100, 100]]


def test_single_step_restarts_the_loop(fake):
    """run() is one step from h (root = the heads' argmax); a loop resumed
    with decode_step after it drafts its first root afresh."""
    s = make_step()
    h = torch.zeros(B, D)
    s.begin_decode(h, False)
    s.decode_step(h, False, mds.GREEDY, 0.0, 0.0)
    s.run(h, mode=mds.GREEDY)
    s.decode_step(h, False, mds.GREEDY, 0.0, 0.0)
    assert fake["tree_root"] == [[7, 7], [7, 7], [7, 7]]
