"""Multi-rank logic on CPU with the gloo backend.

bench.py across ranks (world size 2): each rank runs an independent sequence;
the only cross-rank steps are the barrier and the max-over-ranks timing used
for the whole-job throughput, and the reference arm prints from rank 0 only.

The Ulysses exchanges across ranks (world size 2 and 4): the product's
all-to-all wiring moves each rank's rows to the rank that owns their heads
and the output rows back, checked bit for bit against the single-process
layout and result; the all-gather form gives exactly the all-to-all result.
No GPU needed."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms = 100.0 + 50.0 * rank                      # rank 1 is the slower one
        mx = bench.max_over_ranks(ms, world, "cpu")
        out[rank] = (mx, bench.job_tflops(1e12, 4, world, mx))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo_world2():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for r in (0, 1):
        mx, tf = res[r]
        assert mx == 150.0
        # 2 ranks x 4 steps x 1 TFLOP over the slowest rank's 150 ms
        assert tf == pytest.approx(2 * 4 * 1.0 / 0.150)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5, 1) == 12.5


def test_reference_arm_under_torchrun_prints_once_from_rank0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--workload", "c2", "--steps", "1", "--warmup", "1",
           "--cpu-seconds", "0.1"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["cpu_baseline"]["kind"] == "oracle"
    assert d["unit"] == "TFLOP/s" and d["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] == 0


# ------------------------------------------------ Ulysses exchange across ranks
def _ulysses_worker(rank, world, port, out):
    """Rank `rank` of a Ulysses group of `world` on CPU tensors (gloo).

    The per-token and attention arithmetic are the fp64 oracle's (rounded to
    bf16 where the GPU path stores bf16); what is under test is the product's
    exchange: which rows of which heads reach which rank, in which order."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import torch

    import oracle
    from dit_sequence_attention_gb300 import synth
    from dit_sequence_attention_gb300.ulysses import UlyssesGroup

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        P = world
        S, H, D, kv = 512, 8, 64, 480              # 32 padding keys at the end (in the last rank's shard)
        split = (16, 24, 24)
        S_loc = S // P
        q, k, v = (synth.randn_bf16((S, H, D), 300 + i) for i in range(3))
        wq, wk = synth.norm_weights(D)
        pos = synth.packed_positions(synth.WORKLOADS["tiny"])
        pos = np.concatenate([pos, pos])[:S]         # any position triples will do
        rows = slice(rank * S_loc, (rank + 1) * S_loc)

        def bf16(a):
            return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16)

        def words(t):
            return oracle.bf16_bits(t)

        # this rank's per-token work on its own rows, packed in the exchange's chunk order
        qr = bf16(oracle.norm_rope(oracle.bf16_to_f64(q[rows]), wq.double().numpy(), pos[rows], 1e-6, *split))
        kr = bf16(oracle.norm_rope(oracle.bf16_to_f64(k[rows]), wk.double().numpy(), pos[rows], 1e-6, *split))
        sends = [torch.from_numpy(oracle.seq2head(words(t), P).view(np.int16)).view(torch.bfloat16)
                 for t in (qr, kr, v[rows].contiguous())]
        ug = UlyssesGroup()
        assert (ug.P, ug.rank) == (P, rank)
        recv = [ug.exchange(s) for s in sends]

        # single-process reference: the whole sequence on one rank
        qf = bf16(oracle.norm_rope(oracle.bf16_to_f64(q), wq.double().numpy(), pos, 1e-6, *split))
        kf = bf16(oracle.norm_rope(oracle.bf16_to_f64(k), wk.double().numpy(), pos, 1e-6, *split))
        heads_ok = all(np.array_equal(words(r).reshape(S, H // P, D), oracle.seq2head(words(f), P)[rank])
                       for r, f in zip(recv, (qf, kf, v)))

        # attention of this rank's head group, then the output exchange back to the row owners
        grp = [oracle.bf16_to_f64(r.view(S, H // P, D)) for r in recv]
        o_group = bf16(oracle.attention(*grp, kv_len=kv)).view(P, S_loc, H // P, D)
        o_back = ug.exchange(o_group)
        o_shard = oracle.head2seq(words(o_back), P)
        o_full = bf16(oracle.attention(oracle.bf16_to_f64(qf), oracle.bf16_to_f64(kf), oracle.bf16_to_f64(v),
                                       kv_len=kv))
        out[rank] = (heads_ok, bool(np.array_equal(o_shard, words(o_full)[rows])))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_ulysses_exchange_across_ranks_gloo(world):
    """World size 2 and 4: after the sequence->heads exchange every rank holds
    exactly the single-process seq2head group of its heads (bit for bit), and
    after attention and the heads->sequence exchange every rank holds exactly
    its rows of the single-process output."""
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_ulysses_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert sorted(res) == list(range(world))
    for r in range(world):
        heads_ok, out_ok = res[r]
        assert heads_ok, f"rank {r}: exchanged head-group buffers differ from seq2head of the whole sequence"
        assert out_ok, f"rank {r}: output rows differ from the single-process result"


def test_ulysses_exchange_rejects_mismatched_buffers():
    import torch
    from dit_sequence_attention_gb300.ulysses import _words
    with pytest.raises(ValueError):
        _words(torch.zeros((2, 3), dtype=torch.float32))
    with pytest.raises(ValueError):
        _words(torch.zeros((2, 3), dtype=torch.bfloat16))


# ------------------------------------- all-gather form vs all-to-all form
def _allgather_worker(rank, world, port, out):
    """Rank `rank`: the same step through the two exchange forms of the README
    ("How it works"), the oracle standing in for the kernels.  All-to-all:
    project this rank's rows through all heads, norm/RoPE, exchange, attend,
    exchange back.  All-gather: gather every rank's fp8 hidden rows, project
    all rows through this rank's head rows, norm/RoPE, attend, exchange back."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import torch

    import oracle
    from dit_sequence_attention_gb300 import synth
    from dit_sequence_attention_gb300.ulysses import UlyssesGroup

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        P = world
        S, H, D, hidden, kv = 256, 8, 64, 96, 230
        inner = H * D
        split = (16, 24, 24)
        S_loc = S // P
        rows = slice(rank * S_loc, (rank + 1) * S_loc)
        x = synth.fp8_e4m3_codes((S, hidden), 51, 1.0)
        w = synth.fp8_e4m3_codes((3 * inner, hidden), 52, 4.0)
        scale = 1.0 / (4.0 * hidden ** 0.5)
        wq, wk = synth.norm_weights(D)
        pos = synth.packed_positions(synth.WORKLOADS["tiny"])[:S]
        ug = UlyssesGroup()

        def bf16(a):
            return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16)

        def nr(t, wt, p):
            return bf16(oracle.norm_rope(oracle.bf16_to_f64(t), wt.double().numpy(), p, 1e-6, *split))

        def words(t):
            return oracle.bf16_bits(t)

        def to_bf16_tensor(u16):
            return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16)

        # all-to-all form
        loc = oracle.qkv_proj_fp8(x[rows].numpy(), w.numpy(), scale, inner, 1, 0)        # [S/P, 3, inner]
        q_l, k_l, v_l = (bf16(loc[:, i]).view(S_loc, H, D) for i in range(3))
        q_l, k_l = nr(q_l, wq, pos[rows]), nr(k_l, wk, pos[rows])
        sends = [to_bf16_tensor(oracle.seq2head(words(t), P)) for t in (q_l, k_l, v_l)]
        qa, ka, va = (ug.exchange(s_).view(S, H // P, D) for s_ in sends)

        # all-gather form
        xg = ug.gather_rows(x[rows])
        gathered_ok = torch.equal(xg, x)
        grp = oracle.qkv_proj_fp8(xg.numpy(), w.numpy(), scale, inner, P, rank)          # [S, 3, inner/P]
        qg, kg, vg = (bf16(grp[:, i]).view(S, H // P, D) for i in range(3))
        qg, kg = nr(qg, wq, pos), nr(kg, wk, pos)
        same_inputs = all(torch.equal(a.view(torch.int16), b.view(torch.int16))
                          for a, b in ((qa, qg), (ka, kg), (va, vg)))

        def finish(q_, k_, v_):
            o_g = bf16(oracle.attention(oracle.bf16_to_f64(q_), oracle.bf16_to_f64(k_), oracle.bf16_to_f64(v_),
                                        kv_len=kv)).view(P, S_loc, H // P, D)
            return oracle.head2seq(words(ug.exchange(o_g)), P)

        out[rank] = (gathered_ok, same_inputs, bool(np.array_equal(finish(qa, ka, va), finish(qg, kg, vg))))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_allgather_form_equals_alltoall_form_gloo(world):
    """README "How it works": the all-gather exchange gives exactly the
    all-to-all result.  World size 2 and 4: the gathered hidden rows equal the
    whole hidden state, both forms hand attention bit-identical head-group
    q, k, v, and every rank's output rows are bit-identical."""
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_allgather_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert sorted(res) == list(range(world))
    for r in range(world):
        gathered_ok, same_inputs, same_out = res[r]
        assert gathered_ok, f"rank {r}: gathered hidden rows differ from the whole hidden state"
        assert same_inputs, f"rank {r}: the two forms give attention different q/k/v"
        assert same_out, f"rank {r}: all-gather and all-to-all outputs differ"


def test_ulysses_group_without_process_group():
    """UlyssesGroup(P=, rank=) describes a rank with no process group: its
    compute phases exist, its exchanges refuse; bad ranks and mismatched
    buffers are refused."""
    import torch
    from dit_sequence_attention_gb300.ulysses import UlyssesGroup
    g = UlyssesGroup(P=4, rank=3)
    assert (g.P, g.rank, g.has_group) == (4, 3, False)
    work = g.make_workspace(8, 8, 64, "cpu", hidden=32)
    assert work["qs"].shape == (4, 8, 2, 64) and work["o"].shape == (8, 8, 64) and work["x"].shape == (32, 32)
    assert work["x"].dtype == torch.uint8
    with pytest.raises(RuntimeError):
        g.exchange(work["qs"])
    with pytest.raises(RuntimeError):
        g.gather_rows(torch.zeros((8, 32), dtype=torch.uint8))
    for bad in (-1, 4):
        with pytest.raises(ValueError):
            UlyssesGroup(P=4, rank=bad)


# --------------------------------------------- a rank that fails mid-step
def _failing_peer_worker(rank, world, port, out, mode="exits"):
    """Rank 1 fails before the sequence->heads exchange -- it exits ("exits")
    or stays alive without ever joining the collective ("stalls") -- and
    rank 0, inside the exchange, must get an error (the lost connection, or
    the process group's 5 s timeout) instead of waiting forever."""
    import datetime
    import time

    import torch
    sys.path.insert(0, ROOT)
    from dit_sequence_attention_gb300.ulysses import UlyssesGroup
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=5))
    ug = UlyssesGroup()
    send = torch.zeros((world, 4, 2, 64), dtype=torch.bfloat16)
    if rank == 1:
        out[rank] = "left"
        if mode == "stalls":
            time.sleep(20)                       # alive, but never joins the exchange
        os._exit(0)                              # gone, without a clean shutdown
    t0 = time.monotonic()
    try:
        ug.exchange(send)
        out[rank] = ("no error", time.monotonic() - t0)
    except Exception as e:                       # gloo reports the lost peer or the timeout
        out[rank] = (type(e).__name__, time.monotonic() - t0)
    os._exit(0)


@pytest.mark.parametrize("mode", ["exits", "stalls"])
def test_exchange_with_a_lost_peer_fails_instead_of_hanging(mode):
    port = _free_port()
    ctx = mp.get_context("spawn")
    with mp.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_failing_peer_worker, args=(r, 2, port, out, mode)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        alive = [p for p in procs if p.is_alive()]
        for p in alive:
            p.kill()
        res = dict(out)
    assert not alive, "a rank was still waiting after 120 s"
    assert res.get(1) == "left"
    kind, seconds = res[0]
    assert kind != "no error", "the exchange completed without its peer"
    assert seconds < 15, f"the error took {seconds:.1f} s (process-group timeout 5 s)"
