"""Whole-step parity: MedusaStep (all C-ABI calls in order) against the
oracle's step on the same seeded workload, for the small workloads and the
five benchmark workloads at full size (large batches sampled: the GPU runs
the whole batch, the oracle recomputes some sequences one by one).

A sequence whose draft holds a near-tie (a shortlist or root decision with
oracle margin below the logit tolerance) is compared only up to the draft:
its tree tokens may legitimately differ.  Near-tie acceptance edges end the
comparison of that sequence's path.  Both are counted and printed."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import medusa_synth as ms
import oracle
from tests.gpu_util import (NearTies, check_ranked_ids, close_float, dev, host, require_gpu,
                            tol_logit)
from tests.test_gpu_parity import MINI, MINI_F32, MINI_GQA, f64_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mds():
    require_gpu()
    import speculative_decoding_08_b300 as m
    return m


def make_step(mds, w, x):
    t = {k: dev(x[k], w.dtype) for k in ("W", "lm", "emb", "wqkv", "wo", "kc", "vc")}
    step = mds.MedusaStep(W=t["W"], lm=t["lm"], emb=t["emb"], wqkv=t["wqkv"], wo=t["wo"],
                          Kc=t["kc"], Vc=t["vc"], P=dev(x["P"], "i32"), shortlist=w.shortlist,
                          max_rank_sum=w.max_rank_sum, Hq=w.Hq, Hkv=w.Hkv, B=w.B)
    return step, dev(x["h"], w.dtype)


def compare_step(mds, w, sample, modes):
    x = ms.make_inputs(w)
    step, h = make_step(mds, w, x)
    final_mode = modes[-1]
    results = {}
    for mode in modes:
        commit = mode == final_mode
        step.run(h, mode=0 if mode == "greedy" else 1, eps=w.eps, delta=w.delta, commit=commit)
        torch.cuda.synchronize()
        assert mds.status_check(step.ws) == 0
        results[mode] = dict(L=host(step.L), path=host(step.path), nr=host(step.next_root),
                             ok=host(step.ok).astype(bool))
    g = dict(U=host(step.U), root=host(step.root), topk_id=host(step.topk_id),
             topk_val=host(step.topk_val), tok=host(step.tok), y=host(step.y),
             argmax=host(step.argmax), stats=host(step.stats), child=host(step.childlogit),
             kc=None, vc=None, P=host(step.P))
    f = f64_inputs(w, x, sample)           # h, kc, vc already restricted to the sample
    r = oracle.step(w, f, x["P"][sample], final_mode, batch=list(range(len(sample))))
    ties = NearTies()
    compared_paths = 0
    for i, b in enumerate(sample):
        U = r["U"][i]
        close_float(g["U"][b], U, w.dtype, "stored", f"U[{b}]")
        z = U @ f["lm"].T
        tl = tol_logit(w.dtype, float(np.abs(z).max()))
        n_before = ties.count
        check_ranked_ids([g["root"][b]], z[0], [r["draft"]["root"][i]], tl, ties, f"root[{b}]")
        for k, s in enumerate(w.shortlist):
            check_ranked_ids(g["topk_id"][b, k, :s], z[k + 1], r["draft"]["topk_id"][i, k, :s], tl,
                             ties, f"topk[{b},{k}]")
        if ties.count > n_before:
            continue                       # tree tokens may differ downstream
        np.testing.assert_array_equal(g["tok"][b], r["tok"][i])
        close_float(g["y"][b], r["attn"]["y"][i], w.dtype, "attn", f"y[{b}]")
        st = r["stats"]
        l = r["attn"]["y"][i] @ f["lm"].T
        tv = tol_logit(w.dtype, float(np.abs(l).max()))
        for n in range(r["tree"]["N"]):
            check_ranked_ids([g["argmax"][b, n]], l[n], [st["argmax"][i, n]], tv, ties,
                             f"argmax[{b},{n}]")
        close_float(g["stats"][b, :, 1], st["lse"][i], w.dtype, "logit", "lse")
        close_float(g["stats"][b, :, 2], st["H"][i], w.dtype, "logit", "H")
        close_float(g["child"][b, 1:], st["childlogit"][i, 1:], w.dtype, "logit", "child")
        for mode in modes:
            if mode == final_mode:
                ok, margin, lp = r["ok"], r["margin"], r["path"]
            else:
                ok, margin = oracle.accept_edges(mode, w.eps, w.delta, r["tok"], r["tree"]["parent"], st)
                lp = oracle.longest_path(ok, r["tree"]["parent"], r["tree"]["depth"], st["argmax"], w.K)
            gm = results[mode]
            sure = margin[i] >= tv
            np.testing.assert_array_equal(gm["ok"][b][sure], ok[i][sure])
            if not sure.all():
                ties.add(f"{mode} edge[{b}]")
                continue
            assert gm["L"][b] == lp["L"][i], (mode, b)
            np.testing.assert_array_equal(gm["path"][b], lp["path"][i])
            best = lp["path"][i][lp["L"][i]]
            if st["argmax_gap"][i, best] >= tv:
                assert gm["nr"][b] == lp["next_root"][i]
            compared_paths += 1
            if mode == final_mode:
                # compaction: accepted tree rows moved to P_b..P_b+L, P advanced
                Pb = int(x["P"][b])
                Lb = int(lp["L"][i])
                assert g["P"][b] == Pb + Lb + 1
                kc_g = host(step.Kc[b])
                vc_g = host(step.Vc[b])
                close_float(kc_g[:, Pb:Pb + Lb + 1], r["kc"][i][:, Pb:Pb + Lb + 1], w.dtype,
                            "stored", "kc")
                close_float(vc_g[:, Pb:Pb + Lb + 1], r["vc"][i][:, Pb:Pb + Lb + 1], w.dtype,
                            "stored", "vc")
                np.testing.assert_array_equal(kc_g[:, :Pb], f["kc"][i][:, :Pb])
    ties.report(w.name)
    print(f"[{w.name}] sequences compared: {len(sample)}, paths compared: {compared_paths}, "
          f"near-ties: {ties.count}")
    return ties


SMALL = [(ms.workload(0), ["greedy"]), (MINI, ["greedy", "typical"]), (MINI_GQA, ["typical"]),
         (MINI_F32, ["greedy", "typical"])]


@pytest.mark.parametrize("w,modes", SMALL, ids=lambda p: getattr(p, "name", None))
def test_step_small(mds, w, modes):
    compare_step(mds, w, list(range(w.B)), modes)


FULL = [(1, [0], ["typical"]), (2, [0, 15], ["typical"]), (3, [3], ["typical"]),
        (4, [0, 63], ["greedy", "typical"])]


@pytest.mark.parametrize("cfg,sample,modes", FULL, ids=[f"cfg{c[0]}" for c in FULL])
def test_step_full_size(mds, cfg, sample, modes):
    w = ms.workload(cfg)
    compare_step(mds, w, sample, modes)
    torch.cuda.empty_cache()


def test_captured_step_with_host_buffers(mds):
    """MedusaStep.capture with a pinned host input and host outputs: one graph
    replay reproduces the eager step (h copied in, tokens and path copied out)."""
    w = MINI
    x = ms.make_inputs(w)
    step, h = make_step(mds, w, x)
    step.run(h, mode=1, eps=w.eps, delta=w.delta, commit=False)
    torch.cuda.synchronize()
    want = dict(L=host(step.L), path=host(step.path), tok=host(step.tok), nr=host(step.next_root))
    h_host = h.cpu().pin_memory()
    h_dev = torch.zeros_like(h)
    step.capture(h_dev, mode=1, eps=w.eps, delta=w.delta, commit=False, h_host=h_host,
                 outputs_to_host=True)
    for t in step.host_out.values():
        t.zero_()
    h_dev.zero_()
    step.replay()
    torch.cuda.synchronize()
    assert mds.status_check(step.ws) == 0
    np.testing.assert_array_equal(step.host_out["L"].numpy(), want["L"])
    np.testing.assert_array_equal(step.host_out["path"].numpy(), want["path"])
    np.testing.assert_array_equal(step.host_out["tok"].numpy(), want["tok"])
    np.testing.assert_array_equal(step.host_out["next_root"].numpy(), want["nr"])
    assert torch.equal(h_dev, h)
