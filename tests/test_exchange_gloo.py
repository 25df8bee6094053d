"""The single-GPU layouts against the expert-parallel exchange they stand for.

The multi-source receive layout is the single-GPU shadow of the expert-
parallel exchange.  Two gloo processes stand for two EP ranks, each holding
its own half of a routing.  With its single-source layout, each rank sends
every destination rank the rows of its tokens that reach it (token order)
through one all-to-all.  A destination then holds, source by source, exactly
the rows and token ids of its region in the multi-source layout of the whole
routing.  In the other direction, the combine of the whole routing equals a
reverse all-to-all of the expert-major rows followed by each source's local
weighted sum, bit for bit.  CPU only: the oracle on both sides,
torch.distributed for the exchange."""
import os
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

S = 2                      # source ranks = destination ranks = processes
TS, K, E, H = 37, 3, 8, 16  # tokens per source, top-k, experts (4 per rank), hidden


def _global_inputs():
    sys.path.insert(0, ROOT)
    from combine_moe_dispatch_02_gb300.inputs import random_routing
    idx = random_routing(S * TS, K, E, 321, mask_frac=0.1).numpy()
    x = np.random.default_rng(322).integers(0, 1 << 16, (S * TS, H)).astype(np.uint16)
    return idx, x


def _rank(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, HERE)
    import oracle
    dist.init_process_group("gloo", rank=rank, world_size=S)
    try:
        idx, x = _global_inputs()
        mine = slice(rank * TS, (rank + 1) * TS)
        L = oracle.layout(idx[mine], None, E, S)             # this rank's own tokens, R = S destinations
        # per destination: my tokens that reach it, in token order, as global ids and rows
        send_ids, send_rows, counts = [], [], []
        for r in range(S):
            toks = np.nonzero(L.recv_slot[:, r] >= 0)[0]
            send_ids.append(toks + rank * TS)
            send_rows.append(x[mine][toks])
            counts.append(len(toks))
        cnt_in = torch.empty(S, dtype=torch.int64)
        dist.all_to_all_single(cnt_in, torch.tensor(counts, dtype=torch.int64))
        recv_counts = cnt_in.tolist()
        ids = torch.empty(sum(recv_counts), dtype=torch.int64)
        dist.all_to_all_single(ids, torch.from_numpy(np.concatenate(send_ids).astype(np.int64)),
                               recv_counts, counts)
        rows = torch.empty(sum(recv_counts), H, dtype=torch.int32)          # bf16 patterns, widened for gloo
        dist.all_to_all_single(rows, torch.from_numpy(np.concatenate(send_rows).astype(np.int32)),
                               recv_counts, counts)
        # the multi-source layout of the whole routing, region `rank`
        M = oracle.layout_sources(idx, None, S, E, S)
        n = int(M.tokens_per_rank[rank])
        region = slice(rank * S * TS, rank * S * TS + n)
        recv, st = oracle.dispatch_bf16(x, M)
        ok = (st == 0 and n == len(ids)
              and np.array_equal(M.recv_src_token[region], ids.numpy())
              and np.array_equal(recv[region], rows.numpy().astype(np.uint16))
              and list(M.recv_source_offset[rank]) == [0] + list(np.cumsum(recv_counts)))
        q.put((rank, bool(ok), n))
    except Exception as e:  # reported to the parent
        q.put((rank, repr(e), -1))
    finally:
        dist.destroy_process_group()


def _combine_rank(rank, port, q):
    """Reverse direction: each destination holds the expert-major rows of its
    experts for every source's tokens and sends each source its rows with
    their (token, k); each source then forms the weighted sum locally."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, HERE)
    import oracle
    from combine_moe_dispatch_02_gb300.inputs import bf16_bits, random_weights
    dist.init_process_group("gloo", rank=rank, world_size=S)
    try:
        idx, _ = _global_inputs()
        w = random_weights(S * TS, K, 323).numpy()
        G = oracle.layout(idx, w, E, S)                      # the single-GPU layout of the whole routing
        n_valid = int(G.expert_offset[E])
        y = bf16_bits(torch.randn(n_valid, H, generator=torch.Generator().manual_seed(324)).to(torch.bfloat16))
        out_global, st = oracle.combine(y, G.expert_slot, w)
        m = E // S
        # rows this rank holds: its experts' rows, and the (token, k) each belongs to
        lo, hi = int(G.expert_offset[rank * m]), int(G.expert_offset[(rank + 1) * m])
        owner = np.full((n_valid, 2), -1, np.int64)
        tt, kk = np.nonzero(G.expert_slot >= 0)
        owner[G.expert_slot[tt, kk]] = np.stack([tt, kk], 1)
        send_meta, send_rows, counts = [], [], []
        for src in range(S):
            js = [j for j in range(lo, hi) if owner[j, 0] // TS == src]
            send_meta.append(owner[js].reshape(-1, 2))
            send_rows.append(y[js].reshape(-1, H))
            counts.append(len(js))
        cnt_in = torch.empty(S, dtype=torch.int64)
        dist.all_to_all_single(cnt_in, torch.tensor(counts, dtype=torch.int64))
        rc = cnt_in.tolist()
        meta = torch.empty(sum(rc), 2, dtype=torch.int64)
        dist.all_to_all_single(meta, torch.from_numpy(np.concatenate(send_meta)), rc, counts)
        rows = torch.empty(sum(rc), H, dtype=torch.int32)
        dist.all_to_all_single(rows, torch.from_numpy(np.concatenate(send_rows).astype(np.int32)), rc, counts)
        # local weighted sum over a local slot map of the received rows
        meta = meta.numpy()
        slot_local = np.full((TS, K), -1, np.int32)
        slot_local[meta[:, 0] - rank * TS, meta[:, 1]] = np.arange(len(meta), dtype=np.int32)
        mine = slice(rank * TS, (rank + 1) * TS)
        out_local, st2 = oracle.combine(rows.numpy().astype(np.uint16), slot_local, w[mine])
        ok = (st == 0 and st2 == 0 and len(meta) == int((idx[mine] >= 0).sum())
              and np.array_equal(out_local, out_global[mine]))
        q.put((rank, bool(ok), len(meta)))
    except Exception as e:  # reported to the parent
        q.put((rank, repr(e), -1))
    finally:
        dist.destroy_process_group()


def _run_ranks(target, port_base):
    import oracle
    oracle.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = port_base + os.getpid() % 100
    procs = [ctx.Process(target=target, args=(r, port, q)) for r in range(S)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    return sorted(q.get(timeout=10) for _ in range(S))


def test_combine_matches_a_reverse_exchange_and_local_sum():
    for rank, ok, n in _run_ranks(_combine_rank, 30300):
        assert ok is True, (rank, ok)
        assert n > 0


def test_multi_source_layout_matches_an_all_to_all_exchange():
    for rank, ok, n in _run_ranks(_rank, 30100):
        assert ok is True, (rank, ok)
        assert n > 0
