"""Expert parallelism on CPU ranks: the dispatch plan (native, moe_ep_plan) and
the host side of a layer spread over R ranks (token_dispatch_gb300.ep), with the
MoonEP page's contracts ("Step-by-step"):
  * every rank processes exactly S*K routed rows, whatever the skew;
  * remote experts a rank processes sit in its B = E/R preload slots;
  * reduce_grad adds the slot gradients of every copy into the home expert's
    gradient and clears the slots.
The multi-rank tests run the whole layer on gloo ranks (2 and 4), the expert
arithmetic by the float64 oracle, and compare the layer output and the expert
weight gradients with the oracle's single-process layer on all ranks' tokens."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from token_dispatch_gb300 import _lib as L


def zipf_counts(rng, R, E, S, K, a=1.1):
    """counts [R, E]: each source rank's S tokens choose K distinct experts with
    Zipf-like preferences (the skew of a biased router)."""
    w = 1.0 / np.arange(1, E + 1) ** a
    w = w[rng.permutation(E)]
    w /= w.sum()
    out = np.zeros((R, E), np.int32)
    for r in range(R):
        for _ in range(S):
            out[r, rng.choice(E, K, replace=False, p=w)] += 1
    return out


def check_plan(counts, S, K, B):
    R, E = counts.shape
    G = E // R
    pc, po, se, lc, rr = L.moe_ep_plan(R, E, S, K, B, counts)
    # every destination processes exactly S*K rows
    assert (pc.sum(axis=(1, 2)) == S * K).all()
    # every pair of every bucket (s, e) is processed once: pieces tile the
    # bucket in destination order
    assert (pc.sum(axis=0) == counts).all()
    for s in range(R):
        for e in range(E):
            nxt = 0
            for d in range(R):
                if pc[d, s, e]:
                    assert po[d, s, e] == nxt
                    nxt += pc[d, s, e]
            assert nxt == counts[s, e]
    for d in range(R):
        rows = pc[d].sum(axis=0)  # rows per expert on d
        home = set(range(d * G, (d + 1) * G))
        slots = [int(e) for e in se[d] if e >= 0]
        assert len(slots) == len(set(slots)) <= B
        assert all(e not in home and rows[e] > 0 for e in slots)
        assert (lc[d, :G] == rows[d * G:(d + 1) * G]).all()
        assert [int(v) for v in lc[d, G:G + len(slots)]] == [int(rows[e]) for e in slots]
        # slots hold the remote experts with the most rows; the rest are remote reads
        remote = sorted([(-int(rows[e]), e) for e in range(E) if e not in home and rows[e] > 0])
        assert slots == [e for _, e in remote[:B]]
        assert rr[d] == sum(-c for c, _ in remote[B:])
    return pc, po, se, lc, rr


@pytest.mark.parametrize("R,E,S,K", [(2, 8, 64, 2), (4, 64, 96, 6), (8, 384, 64, 8), (3, 12, 50, 3)])
def test_plan_invariants_under_skew(R, E, S, K):
    rng = np.random.default_rng(R * 1000 + E)
    for a in (0.0, 1.1, 2.5):
        counts = zipf_counts(rng, R, E, S, K, a)
        check_plan(counts, S, K, E // R)
        check_plan(counts, S, K, 2)  # a small pool: the overflow is counted as remote reads


def test_balanced_routing_needs_no_slots():
    R, E, S, K = 4, 16, 40, 2
    G = E // R
    counts = np.zeros((R, E), np.int32)
    for s in range(R):  # source s sends S*K/R pairs to every rank's group, spread evenly
        for d in range(R):
            counts[s, d * G:(d + 1) * G] = S * K // (R * G)
    pc, po, se, lc, rr = check_plan(counts, S, K, G)
    assert (se == -1).all() and (rr == 0).all()
    for d in range(R):  # every rank processes exactly its home group
        assert pc[d][:, :d * G].sum() == 0 and pc[d][:, (d + 1) * G:].sum() == 0


def test_all_pairs_to_one_expert_is_copied_everywhere():
    R, E, S, K = 4, 8, 30, 1
    counts = np.zeros((R, E), np.int32)
    counts[:, 0] = S
    pc, po, se, lc, rr = check_plan(counts, S, K, E // R)
    for d in range(1, R):
        assert se[d, 0] == 0 and lc[d, E // R] == S * K
    assert (rr == 0).all()


def test_plan_rejects_rows_that_do_not_sum_to_SK():
    counts = np.array([[3, 1], [2, 1]], np.int32)  # row 0 sums to 4, row 1 to 3, S*K = 4
    with pytest.raises(L.MoEError):
        L.moe_ep_plan(2, 2, 2, 2, 1, counts)
    with pytest.raises(L.MoEError):
        L.moe_ep_plan(3, 8, 2, 2, 1, np.zeros((3, 8), np.int32))  # E % R != 0


# ------------------------------------------------------------- gloo ranks ---

def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _layer_inputs(R, S, H, E, K, Hp):
    """Seeded inputs of all ranks: tokens [R*S, H], router, experts, dy."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((R * S, H))
    wr = rng.standard_normal((H, E)) * 0.3
    bias = np.zeros(E)
    bias[1] = 1.5  # skew towards expert 1 (rank 0's group)
    wg = rng.standard_normal((E, H, Hp)) / np.sqrt(H)
    wu = rng.standard_normal((E, H, Hp)) / np.sqrt(H)
    wd = rng.standard_normal((E, H, Hp)) / np.sqrt(Hp)
    dy = rng.standard_normal((R * S, H))
    return x, wr, bias, wg, wu, wd, dy


def _rank(rank, world, port, S, H, E, K, Hp, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import oracle as O
    from token_dispatch_gb300 import ep
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x, wr, bias, wg, wu, wd, dy = _layer_inputs(world, S, H, E, K, Hp)
        G = E // world
        mine = slice(rank * S, (rank + 1) * S)
        _, _, idx, gate = O.route(x[mine], wr, K, bias)
        counts = ep.gather_counts(idx, E)
        plan = ep.Plan(counts, S, K, B=G)
        assert int(plan.remote_reads[rank]) == 0
        flat_x = np.repeat(x[mine], K, axis=0)  # row of pair t*K+k is x[t]
        # dispatch: rows to every destination, in its local expert order
        sends = ep.send_rows(plan, rank, idx)
        got = ep.exchange([torch.from_numpy(flat_x[j]) for j in sends],
                          [(int(plan.piece_count[rank, s].sum()), H) for s in range(world)])
        local = ep.assemble(plan, rank, got).numpy()
        n_rows = local.shape[0]
        # local grouped FFN: home experts, then the slot copies
        cu = plan.local_cu_seqlens(rank)
        experts = plan.local_experts(rank)
        h_loc = np.zeros_like(local)
        for i, e in enumerate(experts):
            lo, hi = cu[i], cu[i + 1]
            if hi > lo:
                h_loc[lo:hi] = O.expert_swiglu(local[lo:hi], wg[e], wu[e], wd[e])[1]
        # combine: rows back to their sources, then y = sum_k gate * h
        back = ep.exchange(ep.split_back(plan, rank, torch.from_numpy(h_loc)),
                           [(len(sends[d]), H) for d in range(world)])
        h_pairs = np.zeros((S * K, H))
        for d in range(world):
            h_pairs[sends[d]] = back[d].numpy()
        y = (gate[:, :, None] * h_pairs.reshape(S, K, H)).sum(axis=1)
        # backward: dh of every pair to the rank that computed it, the expert
        # backward there into [G + B] gradient slots, then reduce_grad
        dh_pairs = (gate[:, :, None] * dy[mine][:, None, :]).reshape(S * K, H)
        got_dh = ep.exchange([torch.from_numpy(dh_pairs[j]) for j in sends],
                             [(int(plan.piece_count[rank, s].sum()), H) for s in range(world)])
        dh_loc = ep.assemble(plan, rank, got_dh).numpy()
        grads = torch.zeros((3, G + G, H, Hp), dtype=torch.float64)  # [Wg, Wu, Wd][G + B]
        for i, e in enumerate(experts):
            lo, hi = cu[i], cu[i + 1]
            if hi > lo:
                _, dwg, dwu, dwd = O.expert_swiglu_bwd(local[lo:hi], wg[e], wu[e], wd[e], dh_loc[lo:hi])
                for p, dw in enumerate((dwg, dwu, dwd)):
                    grads[p, i] += torch.from_numpy(dw)
        for p in range(3):
            ep.reduce_grad(plan, grads[p])
        out[rank] = dict(y=y, rows=n_rows, home=grads[:, :G].numpy(), slots_zero=bool((grads[:, G:] == 0).all()),
                         n_slots=int((plan.slot_expert[rank] >= 0).sum()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_expert_parallel_layer_on_gloo_ranks_matches_the_oracle(world):
    import oracle as O
    S, H, E, K, Hp = 24, 16, 8, 2, 12
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, S, H, E, K, Hp, out), nprocs=world, join=True)
        res = dict(out)
    x, wr, bias, wg, wu, wd, dy = _layer_inputs(world, S, H, E, K, Hp)
    G = E // world
    # the single-process layer on all ranks' tokens (routing is per token, so
    # it is the same routing)
    f = O.moe_forward(x, wr, wg, wu, wd, K, bias)
    dh = O.permute_bwd(dy, f["h"], f["gate"], f["dst_row"])[0]
    _, dwg, dwu, dwd = O.expert_ffn_bwd(f["xs"], f["cu"], wg, wu, wd, dh)
    assert any(res[r]["n_slots"] > 0 for r in range(world)), "the skew should need slot copies"
    for r in range(world):
        assert res[r]["rows"] == S * K  # the S x K invariant
        assert np.allclose(res[r]["y"], f["y"][r * S:(r + 1) * S], rtol=1e-12, atol=1e-12)
        for p, ref in enumerate((dwg, dwu, dwd)):
            assert np.allclose(res[r]["home"][p], ref[r * G:(r + 1) * G], rtol=1e-11, atol=1e-12)
        assert res[r]["slots_zero"]
