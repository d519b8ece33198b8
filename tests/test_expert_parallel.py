"""Expert parallelism, host logic on the CPU: the shard ranges, the owner
map, and the two exchange patterns as gloo process groups (world sizes 2 to
4), with each rank's experts computed by the oracle restricted to that
rank's shard (the weights of other ranks' picks set to 0).  The sum over the
ranks must be the whole layer's output (the oracle's, in binary64, within
fp32 rounding of the partial sums), and each rank must receive exactly the
token rows that have one of its experts among their picks."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import oracle  # noqa: E402
import synth  # noqa: E402
from quantized_expert_cache_gb300 import expert_parallel as ep  # noqa: E402

H, F, E, K = 64, 96, 7, 3


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_shard_ranges_partition_every_expert():
    for n_exp in (7, 8, 64, 512, 513):
        for world in (1, 2, 3, 4, 8):
            if world > n_exp:
                continue
            spans = [ep.shard_range(n_exp, r, world) for r in range(world)]
            assert spans[0][0] == 0
            for (b0, n0), (b1, _) in zip(spans, spans[1:]):
                assert b0 + n0 == b1
            assert spans[-1][0] + spans[-1][1] == n_exp
            sizes = [n for _, n in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        ep.shard_range(2, 0, 3)


def test_owners_match_the_ranges():
    for n_exp, world in ((7, 2), (7, 3), (512, 8), (10, 4)):
        ids = torch.arange(n_exp, dtype=torch.int32).reshape(1, -1)
        own = ep.owners(ids, n_exp, world).flatten().tolist()
        for e in range(n_exp):
            b, n = ep.shard_range(n_exp, own[e], world)
            assert b <= e < b + n


def _model():
    wl = synth.Workload("ep", H, E, K, F, 1, routing="zipf", seed=11)
    return wl, [wl.expert_tensor(0, kd) for kd in range(3)]


def _partial(tensors, base, n, x_rows, idx_rows, w_rows):
    """The oracle's layer over this shard's picks only (other picks weigh 0)."""
    idx_np = np.ascontiguousarray(idx_rows, np.int32)
    mine = (idx_np >= base) & (idx_np < base + n)
    wm = np.where(mine, np.asarray(w_rows, np.float64), 0.0)
    if idx_np.shape[0] == 0:
        return np.zeros((0, H))
    return oracle.layer(np.asarray(x_rows, np.float32), idx_np, wm, *tensors, H, F)


def _tokens(wl, rank, T, step=0):
    """Rank `rank`'s own tokens of a step (distinct seeded streams per rank)."""
    if T == 0:
        return np.zeros((0, H), np.float32), np.zeros((0, E), np.float32)
    return wl.x(0, 100 * step + rank, T), wl.logits(0, 100 * step + rank, T)


def _worker(rank, world, port, q, case):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl, tensors = _model()
        base, n = ep.shard_range(E, rank, world)
        if case == "replicated":
            for T in (1, 4):
                x, lg = wl.x(0, 7, T), wl.logits(0, 7, T)  # the same tokens on every rank
                idx, w = oracle.topk(lg, K)
                y = torch.from_numpy(_partial(tensors, base, n, x, idx, w).astype(np.float32))
                ep.allreduce_partial(y)
                y_full = oracle.layer(x, idx, w, *tensors, H, F)
                err = np.abs(y.numpy() - y_full) - (1e-6 + 1e-5 * np.abs(y_full))
                q.put((rank, case, T, float(err.max())))
        else:
            counts = {2: [6, 11], 3: [4, 0, 7], 4: [3, 5, 0, 1]}[world]
            x, lg = _tokens(wl, rank, counts[rank])
            idx, w = oracle.topk(lg, K) if counts[rank] else (np.zeros((0, K), np.int32), np.zeros((0, K)))
            seen = {}

            def local(x_r, idx_r, w_r, step_tokens):
                seen["idx"] = idx_r.numpy().copy()
                seen["step_tokens"] = step_tokens
                return torch.from_numpy(_partial(tensors, base, n, x_r.numpy(), idx_r.numpy(),
                                                 w_r.numpy()).astype(np.float32))

            y, step_tokens = ep.prefill_layer(torch.from_numpy(x), torch.from_numpy(np.asarray(idx, np.int32)),
                                              torch.from_numpy(np.asarray(w, np.float32)), E, local)
            # the rows this rank must have received: every source's tokens
            # with one of its experts among their picks, sources in rank order
            want = []
            for src in range(world):
                xs, ls = _tokens(wl, src, counts[src])
                if counts[src] == 0:
                    continue
                ids, _ = oracle.topk(ls, K)
                for t in range(counts[src]):
                    if ((ids[t] >= base) & (ids[t] < base + n)).any():
                        want.append(ids[t])
            want = np.array(want, np.int32).reshape(-1, K)
            ok_rows = np.array_equal(seen["idx"], want)
            if counts[rank]:
                y_full = oracle.layer(x, idx, w, *tensors, H, F)
                err = float((np.abs(y.numpy() - y_full) - (1e-6 + 1e-5 * np.abs(y_full))).max())
            else:
                err = -1.0 if y.shape == (0, H) else 1.0
            q.put((rank, case, step_tokens == sum(counts) == seen["step_tokens"], ok_rows, err))
    finally:
        dist.destroy_process_group()


def _run(world, case, n_msgs):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q, case)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    return [q.get(timeout=10) for _ in range(n_msgs)]


@pytest.mark.parametrize("world", [2, 3])
def test_replicated_tokens_allreduce_of_partials_is_the_layer(world):
    # synth and the oracle are compiled once before the ranks start
    synth.build()
    oracle.build()
    out = _run(world, "replicated", 2 * world)  # two token counts per rank
    for rank, case, T, err in out:
        assert err <= 0.0, (rank, T, err)


@pytest.mark.parametrize("world", [2, 3, 4])
def test_distributed_tokens_dispatch_and_combine(world):
    synth.build()
    oracle.build()
    out = _run(world, "distributed", world)
    for rank, case, steps_ok, rows_ok, err in out:
        assert steps_ok, rank
        assert rows_ok, rank
        assert err <= 0.0, (rank, err)


def test_rows_forward_passes_rows_and_step_tokens(monkeypatch):
    # the product wrapper around moe_ffn_forward_rows: the received rows, their
    # count and the step's token count reach the library call unchanged
    calls = []

    def fake(ctx, layer, x, n_rows, idx, w, y, step_tokens, stream=None):
        calls.append((ctx, layer, n_rows, step_tokens, tuple(y.shape)))
        y.fill_(1.0)

    monkeypatch.setattr(ep, "moe_ffn_forward_rows", fake)
    run = ep.rows_forward("ctx", 3)
    x = torch.zeros((5, H))
    y = run(x, torch.zeros((5, K), dtype=torch.int32), torch.zeros((5, K)), 17)
    assert calls == [("ctx", 3, 5, 17, (5, H))]
    assert torch.equal(y, torch.ones((5, H)))


def _single_rank(port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=0, world_size=1)
    try:
        wl, tensors = _model()
        x, lg = wl.x(0, 3, 6), wl.logits(0, 3, 6)
        idx, w = oracle.topk(lg, K)

        def local(x_r, idx_r, w_r, st):
            return torch.from_numpy(_partial(tensors, 0, E, x_r.numpy(), idx_r.numpy(), w_r.numpy()).astype(np.float32))

        y, st = ep.prefill_layer(torch.from_numpy(x), torch.from_numpy(np.asarray(idx, np.int32)),
                                 torch.from_numpy(np.asarray(w, np.float32)), E, local)
        y_full = oracle.layer(x, idx, w, *tensors, H, F)
        q.put((st, float((np.abs(y.numpy() - y_full) - (1e-6 + 1e-5 * np.abs(y_full))).max())))
    finally:
        dist.destroy_process_group()


def test_one_rank_is_the_plain_layer():
    # world size 1: every row stays home, the step counts this rank's tokens
    synth.build()
    oracle.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_single_rank, args=(_free_port(), q))
    p.start()
    p.join(120)
    assert p.exitcode == 0
    st, err = q.get(timeout=10)
    assert st == 6 and err <= 0.0



@pytest.mark.parametrize("bad", ["idx", "x", "w"])
def test_dispatch_rejects_other_dtypes(bad):
    # the ids travel as their int32 bits inside one float32 payload row, so a
    # wider id or a half-precision row is refused before any collective
    x, idx, w = torch.zeros((2, H)), torch.zeros((2, K), dtype=torch.int32), torch.zeros((2, K))
    if bad == "idx":
        idx = idx.to(torch.int64)
    elif bad == "x":
        x = x.to(torch.float16)
    else:
        w = w.to(torch.float64)
    with pytest.raises(TypeError):
        ep.dispatch(x, idx, w, E)
