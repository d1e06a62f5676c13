"""Host logic of the unit-sharded path, on CPU: the longest-processing-time partition, the
all-gather of the spectra across gloo ranks (world size 2 and 3), the identical allocation
input on every rank, and a rank that fails before the exchange being seen by its peer."""
import itertools
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import oracle as O
from vlm_compression_fac_b300 import shard


def test_lpt_partition_hand_case_and_determinism():
    parts = shard.lpt_partition([5, 4, 3, 3, 3], 2)
    # 5 -> r0, 4 -> r1, 3 -> r1 (7), 3 -> r0 (8), 3 -> r1 (10)
    assert parts == [[0, 3], [1, 2, 4]]
    assert shard.lpt_partition([5, 4, 3, 3, 3], 2) == parts
    assert shard.lpt_partition([1.0, 1.0, 1.0], 5) == [[0], [1], [2], [], []]
    with pytest.raises(ValueError):
        shard.lpt_partition([1.0], 0)


@pytest.mark.parametrize("seed", range(6))
def test_lpt_partition_is_a_partition_within_the_lpt_bound(seed):
    r = np.random.default_rng(seed)
    k = int(r.integers(3, 9))
    world = int(r.integers(2, 4))
    work = list(r.gamma(1.0, 1.0, k))
    parts = shard.lpt_partition(work, world)
    assert sorted(i for p in parts for i in p) == list(range(k))
    span = max(sum(work[i] for i in p) for p in parts)
    best = min(max(sum(work[i] for i in range(k) if a[i] == q) for q in range(world))
               for a in itertools.product(range(world), repeat=k))
    assert span <= (4.0 / 3.0 - 1.0 / (3.0 * world)) * best + 1e-12


def test_unit_work_orders_the_block_shapes():
    w = {name: shard.unit_work(m, n, 131072) for name, m, n in
         [("q", 4096, 4096), ("k", 4096, 4096), ("gate", 4096, 11008), ("down", 11008, 4096)]}
    assert w["gate"] > w["q"] and w["down"] > w["q"] and w["q"] == w["k"]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _spectra(seed, lens):
    r = np.random.default_rng(seed)
    return [np.sort(r.gamma(1.0, 1.0, n))[::-1].astype(np.float32) for n in lens]


def _gather_worker(rank, world, port, lens, seed, out_q, fail_rank):
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import datetime
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=20))
    try:
        sig = _spectra(seed, lens)
        work = [float(n) ** 3 for n in lens]
        parts = shard.lpt_partition(work, world)
        if rank == fail_rank:
            raise RuntimeError("planted failure before the exchange")
        local = {u: torch.from_numpy(sig[u]) for u in parts[rank]}
        full = shard.gather_spectra(local, lens, parts)
        out_q.put((rank, "ok", full.numpy().tobytes()))
    except Exception as e:  # reported to the parent, which decides what was expected
        out_q.put((rank, "error", repr(e)))
    finally:
        try:
            dist.destroy_process_group()
        except Exception:
            pass


def _run(world, lens, seed, fail_rank=-1):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gather_worker, args=(r, world, port, lens, seed, q, fail_rank)) for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    for _ in range(world):
        rank, status, payload = q.get(timeout=120)
        got[rank] = (status, payload)
    for p in procs:
        p.join(timeout=60)
        if p.is_alive():
            p.kill()
    return got


@pytest.mark.parametrize("world", [2, 3])
def test_gather_spectra_gloo_ranks_agree_and_allocation_is_identical(world):
    lens = [64, 64, 192, 192, 37, 5, 128]
    seed = 40 + world
    got = _run(world, lens, seed)
    sig = _spectra(seed, lens)
    want = np.concatenate(sig)
    costs = [2 * n + 3 for n in lens]
    budget = sum(n * c for n, c in zip(lens, costs)) // 3
    ref = O.allocate(sig, costs, budget, precision="f32")
    for rank in range(world):
        status, payload = got[rank]
        assert status == "ok", payload
        full = np.frombuffer(payload, dtype=np.float32)
        np.testing.assert_array_equal(full, want)
        offs = np.concatenate([[0], np.cumsum(lens)])
        segs = [full[offs[u]:offs[u + 1]] for u in range(len(lens))]
        al = O.allocate(segs, costs, budget, precision="f32")
        np.testing.assert_array_equal(al.ranks, ref.ranks)


def test_a_rank_failing_before_the_exchange_is_seen_by_its_peer():
    got = _run(2, [16, 8, 24], 7, fail_rank=1)
    assert got[1][0] == "error" and "planted failure" in got[1][1]
    assert got[0][0] == "error"   # the all-gather ended with an error instead of waiting forever


def _sharded_worker(rank, world, port, out_q, opts=None):
    import datetime
    import torch
    import torch.distributed as dist
    from synth import recipes
    from tests import cpu_abi_standin as standin
    from vlm_compression_fac_b300 import kfsvd, pipeline
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=60))
    try:
        for name in standin.NAMES:            # this process only: the library calls run on the oracle
            setattr(kfsvd, name, getattr(standin, name))
        ctx = standin._Ctx()
        wl = recipes.mini_block(n_tokens=300, d=64, ffn=96, kv=32, seed=5)
        units = pipeline.unit_specs(wl)
        weights = {}
        for u in wl.units:
            weights.setdefault(u.weight, torch.from_numpy(recipes.gen_full_weight(wl, u)))
        acts = {n: torch.from_numpy(recipes.gen_stream(wl, s, 0, wl.n_tokens)) for n, s in wl.sites.items()
                if s.kind == "act"}
        grads = {n: torch.from_numpy(recipes.gen_stream(wl, s, 0, wl.n_tokens)) for n, s in wl.sites.items()
                 if s.kind == "grad"}
        mine, outs, ranks, cut, used = shard.compress_sharded(ctx, units, weights, acts, grads, wl.n_tokens,
                                                              wl.lam, wl.budget, **(opts or {}))
        prods = {i: (o.U @ o.V).numpy().tobytes() for i, o in zip(mine, outs)}
        out_q.put((rank, "ok", (list(mine), ranks.numpy().tolist(), int(used.item()), prods)))
    except Exception as e:
        out_q.put((rank, "error", repr(e)))
    finally:
        try:
            dist.destroy_process_group()
        except Exception:
            pass


SHARD_OPTS = [None, {"mode": 1}, {"score": "energy_ratio", "unit_weights": [0.5, 1.0, 2.0, 1.5, 0.7, 1.2, 0.9]},
              {"score": "swift_hybrid", "unit_weights": [1.0, 2.0, 0.5, 1.0, 3.0, 1.0, 0.25], "alpha": 0.4}]


@pytest.mark.parametrize("opts", SHARD_OPTS, ids=["half_sigma2", "per_param", "energy_ratio", "swift_hybrid"])
def test_compress_sharded_matches_one_process(monkeypatch, opts):
    """The sharded driver over two gloo ranks, with the library calls replaced by the oracle
    stand-in in each rank: the ranks agree on the allocation, every unit is mapped back by
    exactly one rank, and the result equals the single-process pipeline's, for every
    allocation key the sharded driver offers (the options reach the global allocation; unit
    weights are indexed over all units, not over a rank's share)."""
    import torch
    from synth import recipes
    from tests import cpu_abi_standin as standin
    from vlm_compression_fac_b300 import pipeline
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_sharded_worker, args=(r, 2, port, q, opts)) for r in range(2)]
    for p in procs:
        p.start()
    got = {}
    for _ in range(2):
        rank, status, payload = q.get(timeout=300)
        got[rank] = (status, payload)
    for p in procs:
        p.join(timeout=60)
        if p.is_alive():
            p.kill()
    for r in range(2):
        assert got[r][0] == "ok", got[r][1]
    (m0, r0, u0, p0), (m1, r1, u1, p1) = got[0][1], got[1][1]
    assert r0 == r1 and u0 == u1
    assert sorted(m0 + m1) == list(range(7)) and not set(m0) & set(m1)
    # the same workload in one process
    c = standin.install(monkeypatch)
    wl = recipes.mini_block(n_tokens=300, d=64, ffn=96, kv=32, seed=5)
    units = pipeline.unit_specs(wl)
    weights = {}
    for u in wl.units:
        weights.setdefault(u.weight, torch.from_numpy(recipes.gen_full_weight(wl, u)))
    acts = {n: torch.from_numpy(recipes.gen_stream(wl, s, 0, wl.n_tokens)) for n, s in wl.sites.items()
            if s.kind == "act"}
    grads = {n: torch.from_numpy(recipes.gen_stream(wl, s, 0, wl.n_tokens)) for n, s in wl.sites.items()
             if s.kind == "grad"}
    res = pipeline.compress(c, units, weights, acts, grads, wl.n_tokens, lam=wl.lam, budget=wl.budget,
                            **(opts or {}))
    assert res.ranks.tolist() == r0 and int(res.used.item()) == u0
    prods = dict(p0)
    prods.update(p1)
    for i, o in enumerate(res.units):
        np.testing.assert_array_equal(np.frombuffer(prods[i], dtype=np.float32).reshape(o.m, o.n),
                                      (o.U @ o.V).numpy())


def test_compress_sharded_rejects_what_it_cannot_do():
    from vlm_compression_fac_b300 import shard as S
    with pytest.raises(ValueError):
        S.compress_sharded(None, [], {}, {}, {}, 10, 0.01, 100, score="empirical_fisher")
    with pytest.raises(ValueError):
        S.compress_sharded(None, [object()], {}, {}, {}, 10, 0.01, 100, unit_weights=[1.0, 2.0])
    with pytest.raises(ValueError):
        S.compress_sharded(None, [], {}, {}, {}, 10, 0.01, None)
