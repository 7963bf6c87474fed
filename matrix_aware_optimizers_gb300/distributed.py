"""The optimizer step across ranks: one process per GPU, torch.distributed for the exchange.

Two exchanges, as the pages describe them; every stage of the step itself still runs in
libmao's kernels, and torch.distributed (NCCL on GPUs, gloo in the CPU tests) only moves
bytes between ranks:

* Muon, layer-wise ([Megatron] "レイヤーごとの分散オプティマイザ" and "負荷分散"). Every
  matrix is owned by exactly one rank. The owner is chosen by a cost model, the
  Newton–Schulz flops 4 m^2 n + 2 m^3 per iteration (m <= n), with the longest matrices
  placed first, each on the least-loaded rank, rather than round-robin. Each rank runs
  the whole Muon step (momentum, Newton–Schulz, update) on the matrices it owns; one
  all-gather(v) of the updated weights then gives every rank every matrix.
  The variable-size all-gather needs no copies: the weights live in one byte buffer laid
  out as [rank][that rank's matrices], each rank's segment padded to the largest, so an
  in-place all-gather of the segments is the all-gather(v).

* Sign-Muon ([SignMuon] §2 "Fluxo Algorítmico (Distribuído)", steps 3 and 4). The W_n
  workers are split evenly over the ranks. Each rank packs its workers' signs (one bit per
  entry) into its own rows of a [W_n][stride] word buffer; an in-place all-gather fills the
  other ranks' rows, and every rank then takes the majority vote and applies the update
  locally. The int8 variant (same section, all-reduce variant) sums its local workers'
  int8 signs, exchanges one int8 SUM all-reduce (exact for W_n <= 127) and thresholds the
  sum locally.

The exchange functions take any tensors the process group's backend accepts; the step
functions call the CUDA library and so need CUDA tensors.
"""

from typing import List, Sequence, Tuple

import torch
import torch.distributed as dist

SEGMENT_ALIGN = 256  # bytes: every matrix of a weight segment starts on this boundary


def _before_collective(t: torch.Tensor, group=None) -> None:
    """NCCL orders its collectives after the current stream's work by itself; with gloo and
    CUDA tensors the host must wait for the kernels that produced the data first."""
    if t.is_cuda and dist.is_initialized() and dist.get_backend(group) == "gloo":
        torch.cuda.current_stream(t.device).synchronize()


def _allgather_inplace(flat: torch.Tensor, n: int, rank: int, group=None) -> None:
    """flat = [world][n]: every rank's slice r*n .. r*n + n to every rank, in place."""
    _before_collective(flat, group)
    if flat.is_cuda and dist.get_backend(group) == "gloo":
        parts = list(flat.split(n))
        dist.all_gather(parts, parts[rank].clone(), group=group)
    else:
        dist.all_gather_into_tensor(flat, flat[rank * n:(rank + 1) * n], group=group)


def _rank_world(group=None):
    if dist.is_available() and dist.is_initialized():
        return dist.get_rank(group), dist.get_world_size(group)
    return 0, 1


# ------------------------------------------------------------------ Muon: cost model

def ns_flops(rows: int, cols: int, steps: int = 5) -> int:
    """Newton–Schulz flops of one matrix, (4 m^2 n + 2 m^3) per iteration with m <= n
    ([Megatron] "分散ニュートン・シュルツ": three products per iteration)."""
    m, n = min(rows, cols), max(rows, cols)
    return steps * (4 * m * m * n + 2 * m ** 3)


def assign_lpt(costs: Sequence[float], world: int) -> Tuple[List[int], List[float]]:
    """Owner rank of every unit, longest processing time first: units in decreasing cost
    (ties by index) each go to the rank with the smallest load so far (ties: lowest rank).
    Returns (owners, per-rank loads). Deterministic, so every rank computes the same plan."""
    if world < 1:
        raise ValueError("world size must be >= 1")
    owners = [0] * len(costs)
    loads = [0.0] * world
    for i in sorted(range(len(costs)), key=lambda k: (-costs[k], k)):
        r = min(range(world), key=lambda q: (loads[q], q))
        owners[i] = r
        loads[r] += costs[i]
    return owners, loads


def assign_round_robin(n: int, world: int) -> List[int]:
    """Matrix i on rank i mod world (the plain alternative the cost model replaces)."""
    return [i % world for i in range(n)]


class WeightLayout:
    """Byte layout of a set of weight matrices for the layer-wise exchange:
    [rank][owned matrices of that rank], every matrix 256-byte aligned inside its rank's
    segment, all segments of one size (the largest)."""

    def __init__(self, shapes: Sequence[Tuple[int, int]], dtype: torch.dtype,
                 owners: Sequence[int], world: int):
        if len(shapes) != len(owners):
            raise ValueError("one owner per matrix")
        self.shapes = [tuple(int(v) for v in s) for s in shapes]
        self.dtype = dtype
        self.owners = list(owners)
        self.world = world
        es = torch.empty((), dtype=dtype).element_size()
        self.offset = [0] * len(shapes)   # byte offset inside the owner's segment
        used = [0] * world
        for i, (R, C) in enumerate(self.shapes):
            r = self.owners[i]
            if not 0 <= r < world:
                raise ValueError("owner out of range")
            self.offset[i] = used[r]
            used[r] += (R * C * es + SEGMENT_ALIGN - 1) // SEGMENT_ALIGN * SEGMENT_ALIGN
        self.used = used
        self.segment_bytes = max(max(used), SEGMENT_ALIGN)

    @property
    def total_bytes(self) -> int:
        return self.world * self.segment_bytes

    def allocate(self, device) -> Tuple[torch.Tensor, List[torch.Tensor]]:
        """One zeroed byte buffer and a view per matrix (R x C of the layout's dtype)."""
        flat = torch.zeros(self.total_bytes, dtype=torch.uint8, device=device)
        return flat, self.views(flat)

    def views(self, flat: torch.Tensor) -> List[torch.Tensor]:
        out = []
        for i, (R, C) in enumerate(self.shapes):
            start = self.owners[i] * self.segment_bytes + self.offset[i]
            es = torch.empty((), dtype=self.dtype).element_size()
            out.append(flat[start:start + R * C * es].view(self.dtype).view(R, C))
        return out

    def segment(self, flat: torch.Tensor, rank: int) -> torch.Tensor:
        return flat[rank * self.segment_bytes:(rank + 1) * self.segment_bytes]


def allgather_weights(layout: WeightLayout, flat: torch.Tensor, group=None) -> None:
    """The all-gather(v) of updated weights: every rank's segment to every rank, in place
    (rank r's input is its own segment of the output buffer)."""
    rank, world = _rank_world(group)
    if world != layout.world:
        raise ValueError("layout made for %d ranks, group has %d" % (layout.world, world))
    if world == 1:
        return
    _allgather_inplace(flat, layout.segment_bytes, rank, group)


class LayerwiseMuon:
    """Layer-wise distributed Muon over the ranks of `group`: the owner plan, the weight
    layout, and the step (the owned matrices' muon_step, then the weights' all-gather)."""

    def __init__(self, shapes, w_dtype=torch.bfloat16, steps=5, group=None, balance="lpt"):
        self.group = group
        self.rank, self.world = _rank_world(group)
        self.shapes = [tuple(int(v) for v in s) for s in shapes]
        self.steps = steps
        costs = [ns_flops(R, C, steps) for R, C in self.shapes]
        if balance == "lpt":
            self.owners, self.loads = assign_lpt(costs, self.world)
        elif balance == "round_robin":
            self.owners = assign_round_robin(len(costs), self.world)
            self.loads = [0.0] * self.world
            for i, r in enumerate(self.owners):
                self.loads[r] += costs[i]
        else:
            raise ValueError(balance)
        self.mine = [i for i, r in enumerate(self.owners) if r == self.rank]
        self.layout = WeightLayout(self.shapes, w_dtype, self.owners, self.world)

    def imbalance(self) -> float:
        """Largest rank load over the mean load (1.0 is perfect balance)."""
        mean = sum(self.loads) / self.world
        return max(self.loads) / mean if mean > 0 else 1.0

    def step(self, W: Sequence[torch.Tensor], M_own, G_own, mu, lr, steps=5, coeffs=None,
             eps=1e-7, ws=None, flat=None, stream=None):
        """One step: muon_step on the owned matrices (W[i] for i in self.mine, with their
        momenta M_own and gradients G_own in the same order), then the all-gather of the
        updated weights. W must be the views of `flat` (WeightLayout.allocate)."""
        import matrix_aware_optimizers_gb300 as mao
        if flat is None:
            raise ValueError("the weights' byte buffer (WeightLayout.allocate) is required")
        if len(M_own) != len(self.mine) or len(G_own) != len(self.mine):
            raise ValueError("one momentum and one gradient per owned matrix")
        if self.mine:
            mao.muon_step([W[i] for i in self.mine], list(M_own), list(G_own), mu, lr,
                          steps=steps, coeffs=coeffs if coeffs is not None else mao.QUINTIC,
                          eps=eps, ws=ws, stream=stream)
        allgather_weights(self.layout, flat, self.group)


# ------------------------------------------------------------------ Sign-Muon

class SignExchange:
    """The [W_n][stride] buffers of the Sign-Muon exchange for one R x C matrix, with the
    W_n workers split evenly over the ranks (rank r holds workers r*L .. r*L + L - 1)."""

    def __init__(self, rows, cols, workers, group=None):
        self.group = group
        self.rank, self.world = _rank_world(group)
        if workers % self.world:
            raise ValueError("%d workers do not split evenly over %d ranks" % (workers, self.world))
        self.rows, self.cols, self.workers = int(rows), int(cols), int(workers)
        self.local = workers // self.world
        self.nbits = self.rows * self.cols
        self.nwords = (self.nbits + 31) // 32
        self.stride = (self.nwords + 3) // 4 * 4          # words: 16-byte aligned rows
        self.s_stride = (self.nbits + 15) // 16 * 16      # int8 entries: 16-byte aligned

    @property
    def first_worker(self) -> int:
        return self.rank * self.local

    def allocate_words(self, device) -> torch.Tensor:
        return torch.zeros((self.workers, self.stride), dtype=torch.int32, device=device)

    def my_words(self, words: torch.Tensor) -> List[torch.Tensor]:
        """This rank's workers' rows (each ceil(R*C/32) words)."""
        w0 = self.first_worker
        return [words[w0 + k, :self.nwords] for k in range(self.local)]

    def allgather_words(self, words: torch.Tensor) -> None:
        """1-bit all-gather ([SignMuon] §2 step 3): every rank's rows to every rank."""
        if self.world == 1:
            return
        _allgather_inplace(words.view(-1), self.local * self.stride, self.rank, self.group)

    def allreduce_int8(self, partial: torch.Tensor) -> None:
        """int8 SUM all-reduce ([SignMuon] §2 step 3, all-reduce variant) of a partial sum of
        signs; exact while the total number of workers is at most 127."""
        if self.workers > 127:
            raise ValueError("the int8 sum of more than 127 signs can wrap")
        if self.world > 1:
            _before_collective(partial, self.group)
            dist.all_reduce(partial, op=dist.ReduceOp.SUM, group=self.group)


def sign_muon_step(ex: SignExchange, W, M_local, G_local, words, vote, mu, lr, steps=5,
                   coeffs=None, eps=1e-7, compute="bf16", ws=None, stream=None):
    """One Sign-Muon step of this rank ([SignMuon] §2 steps 1-4, all-gather variant): local
    momentum and Newton–Schulz of its workers with the signs packed into its rows of
    `words`, the all-gather of the packed rows, then the vote and the update of W, which
    every rank applies identically."""
    import matrix_aware_optimizers_gb300 as mao
    co = coeffs if coeffs is not None else mao.QUINTIC
    mao.muon_momentum_update(M_local, G_local, mu, stream=stream)
    mao.ns_orthogonalize(M_local, None, steps, co, eps, compute, sign_bits=ex.my_words(words),
                         ws=ws, stream=stream)
    ex.allgather_words(words)
    mao.majority_vote_packed(words, ex.nbits, vote, stream=stream)
    mao.apply_update(W, lr, vote=vote, stream=stream)


def sign_muon_step_int8(ex: SignExchange, W, M_local, G_local, U_local, s8_local, total, vote,
                        mu, lr, steps=5, coeffs=None, eps=1e-7, compute="bf16", ws=None,
                        stream=None):
    """One Sign-Muon step of this rank, int8 all-reduce variant: local momentum and
    Newton–Schulz, int8 signs of its workers into s8_local ([L][stride] int8), their local
    sum into `total` (int8, R*C), the SUM all-reduce of `total`, then the threshold (a tie
    gives +1) packed into `vote` and the update of W."""
    import matrix_aware_optimizers_gb300 as mao
    co = coeffs if coeffs is not None else mao.QUINTIC
    mao.muon_momentum_update(M_local, G_local, mu, stream=stream)
    mao.ns_orthogonalize(M_local, U_local, steps, co, eps, compute, ws=ws, stream=stream)
    for k in range(ex.local):
        mao.sign_int8(U_local[k], s8_local[k, :ex.nbits].view(ex.rows, ex.cols), stream=stream)
    mao.majority_vote_int8(s8_local, ex.nbits, sum=total, stream=stream)
    ex.allreduce_int8(total)
    # the all-reduced sum is one "worker" holding sum_m S^(m): its threshold is the vote
    mao.majority_vote_int8(total.view(1, -1), ex.nbits, vote=vote, stream=stream)
    mao.apply_update(W, lr, vote=vote, stream=stream)
