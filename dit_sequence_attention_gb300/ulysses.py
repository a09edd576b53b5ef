"""Ulysses sequence parallelism across ranks: the all-to-all and all-gather forms.

"buqi-minimax-h3-multigpu" README, "How it works": every rank keeps a
row-shard of the packed sequence for the per-token work (QK-norm, RoPE); for
attention an all-to-all regroups q, k and v so that each rank holds every row
of 56/P heads, the rank evaluates exact attention for those heads, and a
second all-to-all returns the output rows to their owners.

Rank r of a group of P holds rows [r*S/P, (r+1)*S/P) of the packed sequence.
Its per-token kernels write the send buffer directly in the exchange's order:
``h3attn_qk_norm_rope_seq2head`` / ``h3attn_seq2head`` with degree P applied to
the local shard give ``send[g] = shard[:, g*H/P:(g+1)*H/P]`` ([P][S/P][H/P][D]),
the rows of head group g that rank g needs.  One ``all_to_all_single`` moves
chunk g to rank g; what arrives is ``recv[src] = rows of rank src for this
rank's heads``, i.e. the head-group buffer [S][H/P][D] in global row order,
which ``h3attn_forward`` reads as it is (no unpack).  The output goes back
through the same exchange: the group output [S][H/P][D] seen as
[P][S/P][H/P][D] sends rank g its own rows, and ``h3attn_head2seq`` of what
arrives gives this rank's [S/P][H][D] output shard.

The all-gather variant (same README section: for world sizes up to 4 the
modulated hidden state is gathered instead, and every rank projects all rows
through only its own head rows of qkv_proj -- exact because the fp8 weight has
one scale per tensor): ``gather_rows`` collects the fp8 hidden rows of every
rank, ``project`` runs ``h3attn_qkv_proj_fp8`` for this rank's heads straight
into the head-group buffers, ``norm_rope_group`` applies the QK-norm and RoPE
there (per token and head, so with all rows' positions), and attention and the
output exchange follow as in the all-to-all form.  Both forms give
bit-identical outputs: the projection of one (row, output column) and the
per-row norm / rotation / attention do not depend on how rows and heads are
split.

The exchanges move whole bf16 rows as 32-bit words (bit-exact; the element
types every backend supports), with NCCL on GPUs and gloo on CPU tensors.
Every buffer handed to a collective is memory of this rank's own device; the
collectives are plain point-to-point transfers (set ``NCCL_NVLS_ENABLE=0`` before the
process group is created).
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def _words(t: torch.Tensor) -> torch.Tensor:
    """The bf16 tensor's bits as int32 words (pairs of adjacent bf16 values)."""
    if t.dtype != torch.bfloat16 or not t.is_contiguous() or t.shape[-1] % 2:
        raise ValueError("exchange buffers must be contiguous bf16 with an even last dimension")
    return t.view(torch.int32)


class UlyssesGroup:
    """One rank of a Ulysses group of P ranks.

    ``UlyssesGroup(group)`` takes P and the rank from a torch.distributed
    process group (None: the default group).  ``UlyssesGroup(P=..., rank=...)``
    describes a rank without a process group: its pack / attend / unpack
    phases run, and ``exchange`` refuses (there is nobody to exchange with).
    """

    def __init__(self, group=None, *, P: int | None = None, rank: int | None = None):
        self.group = group
        self.has_group = P is None
        if self.has_group:
            self.P = dist.get_world_size(group)
            self.rank = dist.get_rank(group)
        else:
            if rank is None or not 0 <= rank < P:
                raise ValueError("an explicit P needs a rank in [0, P)")
            self.P, self.rank = int(P), int(rank)

    def exchange(self, send: torch.Tensor, recv: torch.Tensor | None = None) -> torch.Tensor:
        """All-to-all of [P][rows][H/P][D] bf16 chunks: chunk g of `send` goes to
        rank g and arrives there as chunk `self.rank` of its `recv`.

        Sequence -> heads: send = this rank's rows split by head group; recv =
        every rank's rows of this rank's head group ([S][H/P][D] in row order).
        Heads -> sequence: send = this rank's head-group output [S][H/P][D];
        recv[g] = this rank's rows of head group g.
        """
        if not self.has_group:
            raise RuntimeError("this UlyssesGroup was made without a process group; it cannot exchange")
        if send.shape[0] != self.P:
            raise ValueError(f"send must have {self.P} chunks along dim 0, got shape {tuple(send.shape)}")
        if recv is None:
            recv = torch.empty_like(send)
        elif recv.shape != send.shape or recv.dtype != send.dtype or recv.device != send.device:
            raise ValueError("recv must match send in shape, dtype and device")
        dist.all_to_all_single(_words(recv), _words(send), group=self.group)
        return recv

    def make_workspace(self, S_local: int, H: int, D: int, device, hidden: int | None = None) -> dict:
        """Buffers of one distributed step (allocated once by the caller);
        `hidden` adds the gathered fp8 hidden state of the all-gather form."""
        P = self.P
        e = dict(dtype=torch.bfloat16, device=device)
        shape = (P, S_local, H // P, D)
        work = {name: torch.empty(shape, **e) for name in ("qs", "ks", "vs", "qh", "kh", "vh", "oh", "os")}
        work["o"] = torch.empty((S_local, H, D), **e)
        if hidden is not None:
            work["x"] = torch.empty((P * S_local, hidden), dtype=torch.uint8, device=device)
        return work

    def gather_rows(self, x_local: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
        """All-gather of this rank's rows [S/P][...] into [S][...] in rank order
        (the fp8 hidden state of the all-gather form, as uint8 codes)."""
        if not self.has_group:
            raise RuntimeError("this UlyssesGroup was made without a process group; it cannot exchange")
        x_local = x_local.contiguous()
        if out is None:
            out = torch.empty((self.P * x_local.shape[0],) + tuple(x_local.shape[1:]), dtype=x_local.dtype,
                              device=x_local.device)
        elif out.shape[0] != self.P * x_local.shape[0] or out.shape[1:] != x_local.shape[1:] or \
                out.dtype != x_local.dtype or out.device != x_local.device:
            raise ValueError("out must be [P * rows, ...] of the same dtype and device as x_local")
        dist.all_gather_into_tensor(out, x_local, group=self.group)
        return out

    def pack(self, q, k, v, w_q, w_k, pos, d_t, d_h, d_w, eps, theta, work, stream):
        """Per-token work on this rank's rows, written in the exchange's chunk
        order: QK-norm + RoPE of q and k, and v, each as [P][S/P][H/P][D]."""
        from . import h3attn_qk_norm_rope_seq2head, h3attn_seq2head
        h3attn_qk_norm_rope_seq2head(q, k, work["qs"], work["ks"], w_q, w_k, pos, self.P, d_t, d_h, d_w, eps, theta,
                                     stream=stream)
        h3attn_seq2head(v, work["vs"], self.P, stream)

    def project(self, x_full, w_fp8, scale, work, stream):
        """All-gather form: q, k, v of this rank's heads for every row, as the
        head-group buffers [S][H/P][D]: the gathered hidden state [S][hidden]
        (E4M3 codes) through this rank's head rows of qkv_proj
        ([3 * inner][hidden] E4M3, q then k then v rows), times `scale`."""
        from . import h3attn_qkv_proj_fp8
        h3attn_qkv_proj_fp8(x_full, w_fp8, scale, work["qh"], work["kh"], work["vh"], self.P, self.rank,
                            stream=stream)

    def norm_rope_group(self, w_q, w_k, pos, d_t, d_h, d_w, eps, theta, work, stream):
        """All-gather form: QK-norm and RoPE in place on the head-group buffers
        (every row, this rank's heads; `pos` holds all S rows' positions)."""
        from . import h3attn_qk_norm_rope
        P, S_loc, Hp, D = work["qh"].shape
        grp = lambda t: t.view(P * S_loc, Hp, D)
        h3attn_qk_norm_rope(grp(work["qh"]), grp(work["kh"]), grp(work["qh"]), grp(work["kh"]), w_q, w_k, pos,
                            d_t, d_h, d_w, eps, theta, stream=stream)

    def attend(self, kv_len, work, stream):
        """Exact attention of this rank's head group over the whole sequence
        (the received [S][H/P][D] buffers, in global row order)."""
        from . import h3attn_forward
        P, S_loc, Hp, D = work["qh"].shape
        grp = lambda t: t.view(P * S_loc, Hp, D)
        h3attn_forward(grp(work["qh"]), grp(work["kh"]), grp(work["vh"]), grp(work["oh"]), kv_len=kv_len,
                       stream=stream)

    def unpack(self, work, stream):
        """This rank's output rows [S/P][H][D] from the returned chunks."""
        from . import h3attn_head2seq
        h3attn_head2seq(work["os"], work["o"], self.P, stream)
        return work["o"]

    def attention_step(self, q, k, v, w_q, w_k, pos, kv_len, d_t, d_h, d_w, eps=1e-6, theta=10000.0,
                       work=None, stream=None):
        """One Ulysses attention step of this rank.

        q, k, v  [S/P][H][D] bf16: this rank's rows of the packed sequence.
        pos      [S/P][3] int32: the positions of those rows.
        kv_len   valid keys of the WHOLE sequence (keys >= kv_len are padding).
        Returns this rank's output rows [S/P][H][D].  Requires H % P == 0 and
        (S/P) % P == 0 (the per-rank pack splits the shard's rows into P
        equal chunks of the exchange).
        """
        P = self.P
        S_loc, H, D = q.shape
        if H % P or S_loc % P:
            raise ValueError(f"P={P} must divide H={H} and the shard length S/P={S_loc}")
        if work is None:
            work = self.make_workspace(S_loc, H, D, q.device)
        if stream is None:
            stream = torch.cuda.current_stream(q.device)
        self.pack(q, k, v, w_q, w_k, pos, d_t, d_h, d_w, eps, theta, work, stream)
        with torch.cuda.stream(stream):
            for src, dst in (("qs", "qh"), ("ks", "kh"), ("vs", "vh")):
                self.exchange(work[src], work[dst])
        self.attend(kv_len, work, stream)
        with torch.cuda.stream(stream):
            self.exchange(work["oh"], work["os"])
        return self.unpack(work, stream)

    def attention_step_allgather(self, x_local, w_fp8, scale, w_q, w_k, pos, kv_len, d_t, d_h, d_w, eps=1e-6,
                                 theta=10000.0, work=None, stream=None):
        """One step of this rank in the all-gather form.

        x_local  [S/P][hidden] E4M3 codes (uint8): this rank's rows of the
                 modulated hidden state.
        w_fp8    [3 * H * D][hidden] E4M3 codes of qkv_proj; `scale` the
                 product of the two per-tensor scales.
        pos      [S][3] int32: the positions of ALL rows (every rank computes
                 attention over the whole sequence for its heads).
        kv_len   valid keys of the whole sequence.
        Returns this rank's output rows [S/P][H][D], bit-identical to the
        all-to-all form fed with the same projection.
        """
        P = self.P
        S_loc, hidden = x_local.shape
        inner = w_fp8.shape[0] // 3
        D = w_q.numel()
        H = inner // D
        if inner % D or H % P or S_loc % P:
            raise ValueError(f"P={P} must divide H={H} and the shard length S/P={S_loc}")
        if work is None:
            work = self.make_workspace(S_loc, H, D, x_local.device, hidden=hidden)
        elif "x" not in work:
            raise ValueError("the workspace of the all-gather form needs make_workspace(..., hidden=...)")
        if stream is None:
            stream = torch.cuda.current_stream(x_local.device)
        with torch.cuda.stream(stream):
            self.gather_rows(x_local, work["x"])
        self.project(work["x"], w_fp8, scale, work, stream)
        self.norm_rope_group(w_q, w_k, pos, d_t, d_h, d_w, eps, theta, work, stream)
        self.attend(kv_len, work, stream)
        with torch.cuda.stream(stream):
            self.exchange(work["oh"], work["os"])
        return self.unpack(work, stream)
