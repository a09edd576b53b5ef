"""The distributed Ulysses step on the GPU.

Across ranks the step is: per-token work on each rank's rows written in the
exchange's chunk order, an all-to-all of q', k', v, attention of each rank's
head group, an all-to-all of the output, and the unpack to each rank's rows.
One GPU cannot host several ranks whose collectives wait on one another, so
(1) P ranks are emulated in one process by running each rank's phases on the
GPU with the all-to-all done as plain device copies (chunk g of rank r's send
buffer -> chunk r of rank g's receive buffer), and the assembled output must
equal the single-GPU step bit for bit; (2) the real collective path (both the all-to-all and the all-gather form)
runs as a one-rank NCCL group in a child process.  The all-gather form on
emulated ranks is checked bit for bit against the same single-GPU step.  The multi-rank collective wiring
itself is tested on CPU with gloo (world size 2 and 4)."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from conftest import ROOT
from dit_sequence_attention_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h3(cuda_device):
    from dit_sequence_attention_gb300 import build
    build.build()
    import dit_sequence_attention_gb300 as m
    m.load_library()
    return m


@pytest.mark.parametrize("P", [2, 4, 8])
def test_rank_phases_with_emulated_exchange_equal_the_single_gpu_step(h3, cuda_device, P):
    from dit_sequence_attention_gb300.ulysses import UlyssesGroup
    w = synth.WORKLOADS["c2"]
    dev = cuda_device
    q, k, v = synth.qkv(w, dev)
    wq, wk = (t.to(dev) for t in synth.norm_weights(w.D))
    pos = torch.from_numpy(synth.packed_positions(w)).to(dev)
    S_loc = w.S // P
    stream = torch.cuda.current_stream(dev)
    ranks = [UlyssesGroup(P=P, rank=r) for r in range(P)]
    works = [g.make_workspace(S_loc, w.H, w.D, dev) for g in ranks]
    for r, g in enumerate(ranks):
        rows = slice(r * S_loc, (r + 1) * S_loc)
        g.pack(q[rows].contiguous(), k[rows].contiguous(), v[rows].contiguous(), wq, wk, pos[rows].contiguous(),
               *w.rope_split, w.eps, w.theta, works[r], stream)
    for r in range(P):                      # sequence -> heads
        for src in range(P):
            for a, b in (("qs", "qh"), ("ks", "kh"), ("vs", "vh")):
                works[r][b][src].copy_(works[src][a][r])
    for r, g in enumerate(ranks):
        g.attend(w.S_v, works[r], stream)
    for r in range(P):                      # heads -> sequence
        for src in range(P):
            works[r]["os"][src].copy_(works[src]["oh"][r])
    out = torch.cat([g.unpack(works[r], stream) for r, g in enumerate(ranks)])
    ref = h3.ulysses_attention_step(q, k, v, wq, wk, pos, P, w.S_v, *w.rope_split, w.eps, w.theta)
    torch.cuda.synchronize()
    assert h3.h3attn_get_device_status() == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("P", [2, 4])
def test_allgather_form_with_emulated_exchange_equals_the_single_gpu_step(h3, cuda_device, P):
    """The all-gather form on P emulated ranks -- each rank projects the whole
    gathered fp8 hidden state through its own head rows of qkv_proj, applies
    QK-norm and RoPE to its head group, attends, and the output exchange is done
    as device copies -- equals the single-GPU step on the full projection bit
    for bit ("ag vs a2a exact" in the README's terms)."""
    from dit_sequence_attention_gb300.ulysses import UlyssesGroup
    w = synth.WORKLOADS["c2"]
    dev = cuda_device
    hidden, inner = synth.HIDDEN, synth.INNER
    x = synth.fp8_e4m3_codes((w.S, hidden), 61, 1.0, dev)
    wt = synth.fp8_e4m3_codes((3 * inner, hidden), 62, 4.0, dev)
    scale = 1.0 / (4.0 * hidden ** 0.5)
    wq, wk = (t.to(dev) for t in synth.norm_weights(w.D))
    pos = torch.from_numpy(synth.packed_positions(w)).to(dev)
    q, k, v = (torch.empty((w.S, w.H, w.D), dtype=torch.bfloat16, device=dev) for _ in range(3))
    h3.h3attn_qkv_proj_fp8(x, wt, scale, q, k, v, 1, 0)
    ref = h3.ulysses_attention_step(q, k, v, wq, wk, pos, P, w.S_v, *w.rope_split, w.eps, w.theta).clone()
    S_loc = w.S // P
    stream = torch.cuda.current_stream(dev)
    ranks = [UlyssesGroup(P=P, rank=r) for r in range(P)]
    works = [g.make_workspace(S_loc, w.H, w.D, dev) for g in ranks]
    for r, g in enumerate(ranks):
        g.project(x, wt, scale, works[r], stream)   # every rank receives the whole hidden state
        g.norm_rope_group(wq, wk, pos, *w.rope_split, w.eps, w.theta, works[r], stream)
        g.attend(w.S_v, works[r], stream)
    for r in range(P):                      # heads -> sequence
        for src in range(P):
            works[r]["os"][src].copy_(works[src]["oh"][r])
    out = torch.cat([g.unpack(works[r], stream) for r, g in enumerate(ranks)])
    torch.cuda.synchronize()
    assert h3.h3attn_get_device_status() == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


_ONE_RANK = r"""
import os, sys, socket, datetime
sys.path.insert(0, sys.argv[1])
import numpy as np, torch, torch.distributed as dist
import dit_sequence_attention_gb300 as h3
from dit_sequence_attention_gb300 import synth
from dit_sequence_attention_gb300.ulysses import UlyssesGroup
with socket.socket() as s:
    s.bind(("127.0.0.1", 0)); port = s.getsockname()[1]
torch.cuda.set_device(0)
dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                        timeout=datetime.timedelta(seconds=120))
try:
    w = synth.WORKLOADS["c2"]
    dev = torch.device("cuda:0")
    q, k, v = synth.qkv(w, dev)
    wq, wk = (t.to(dev) for t in synth.norm_weights(w.D))
    pos = torch.from_numpy(synth.packed_positions(w)).to(dev)
    g = UlyssesGroup()
    o = g.attention_step(q, k, v, wq, wk, pos, w.S_v, *w.rope_split, w.eps, w.theta).clone()
    ref = h3.ulysses_attention_step(q, k, v, wq, wk, pos, 1, w.S_v, *w.rope_split, w.eps, w.theta)
    torch.cuda.synchronize()
    assert h3.h3attn_get_device_status() == 0
    assert torch.equal(o.view(torch.int16), ref.view(torch.int16)), "one-rank group differs from the step"
    hidden, inner = synth.HIDDEN, synth.INNER
    x = synth.fp8_e4m3_codes((w.S, hidden), 61, 1.0, dev)
    wt = synth.fp8_e4m3_codes((3 * inner, hidden), 62, 4.0, dev)
    scale = 1.0 / (4.0 * hidden ** 0.5)
    o_ag = g.attention_step_allgather(x, wt, scale, wq, wk, pos, w.S_v, *w.rope_split, w.eps, w.theta).clone()
    qp, kp, vp = (torch.empty((w.S, w.H, w.D), dtype=torch.bfloat16, device=dev) for _ in range(3))
    h3.h3attn_qkv_proj_fp8(x, wt, scale, qp, kp, vp, 1, 0)
    ref_ag = h3.ulysses_attention_step(qp, kp, vp, wq, wk, pos, 1, w.S_v, *w.rope_split, w.eps, w.theta)
    torch.cuda.synchronize()
    assert h3.h3attn_get_device_status() == 0
    assert torch.equal(o_ag.view(torch.int16), ref_ag.view(torch.int16)), "all-gather form differs from the step"
    print("ONE_RANK_OK")
finally:
    dist.destroy_process_group()
"""


def test_one_rank_nccl_group_runs_the_collective_path(h3, cuda_device):
    env = dict(os.environ, NCCL_NVLS_ENABLE="0", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, "-c", _ONE_RANK, ROOT], capture_output=True, text=True, timeout=300,
                       env=env, cwd=ROOT)
    assert r.returncode == 0 and "ONE_RANK_OK" in r.stdout, (r.stdout[-2000:], r.stderr[-3000:])
