"""Plain fp64 CPU oracle of the Muon / Sign-Muon optimizer step.

TEST INFRASTRUCTURE. Only the test suite (``tests/``), ``__graft_entry__.smoke()``
and the CPU-baseline / reference legs of ``bench.py`` may import this package.
The product (the CUDA library ``libmao.so`` and its Python binding in
``matrix_aware_optimizers_gb300``) never imports, links or executes anything
here, and this package imports nothing from the product: the two share no
kernels, helpers, tables or constants. Inputs reach both sides from the seeded
generators in ``matrix_aware_optimizers_gb300.workloads`` (random draws only,
none of the method's arithmetic).

The code is deliberately slow and literal: numpy fp64 for floating point,
plain Python loops for the small bit-level cases, library matmuls as steps, and
no blocking, fusion or reordering beyond what the sources state.

Sources, cited by page title and section:

  [SignMuon]  "Resumo Técnico: SignMuon: Otimização Distribuída de Muon com
              Eficiência de Comunicação" (gist.science, paper 2605.16311).
  [Megatron]  "NVIDIA MegatronによるLLM学習高速化へ向けた新世代オプティマイザの高度化"
              (news.ainew.jp).
  [Dion]      "대규모 AI 모델 학습을 10배 빠르게: Dion 옵티마이저를 사용한 분산 학습"
              (dsdanielpark.github.io).

Parity pins (every function below is checked by ``tests/test_oracle_pins.py``
against something other than itself):

  rounding.bf16_rne        hand-computed table (tests/golden/bf16_rne.txt) + torch CPU cast
  rounding.fma_f32         exact Fraction arithmetic with an independent rounding rule,
                           and hand-built double-rounding traps
  muon.momentum            follows from fma_f32 / bf16_rne pins + a hand table
  muon.newton_schulz       SVD closed form (odd polynomial acts on singular values),
                           cubic convergence to scipy's polar factor, invariants
  muon.blockwise_newton_schulz  1 x 1 grid = newton_schulz; block independence; on a
                           block-diagonal input the cubic iteration reaches scipy's polar
                           factor of the whole matrix
  muon.sign_of/pack_signs  hand-computed words (tests/golden/pack_signs.txt)
  muon.majority_vote       exhaustive brute force over all sign patterns (W_n <= 8)
  muon.int8_sum_vote       brute-force integer sums; equals the packed-bit vote on all patterns
  muon.post_vote_polar     Newton-Schulz pins (it is newton_schulz on the +-1 matrix)
  muon.apply_update        hand-computed rounding table (tests/golden/update_rounding.txt)
  muon.sign_muon_step      composition checked against an SVD-route recomputation
  dion.orthonormalise_columns  classical Gram-Schmidt loop; P = Q R with R upper triangular
  dion.column_normalize    unit column norms, directions kept, zero columns
  dion.dion_step           exact rank-r buffer with Q_prev = its right singular vectors gives
                           the polar factor U V^T; full rank gives M = mu B; error feedback
                           M + (1 - mu) P R^T = B

No function is "parity unpinned".
"""

from .rounding import bf16_rne, fma_f32, to_f32
from .dion import column_normalize, dion_step, orthonormalise_columns
from .muon import (
    QUINTIC,
    CUBIC,
    momentum,
    frobenius_normalise,
    newton_schulz,
    blockwise_newton_schulz,
    sign_of,
    pack_signs,
    pack_signs_loop,
    unpack_signs,
    majority_vote,
    int8_sum_vote,
    post_vote_polar,
    apply_update,
    apply_update_f64,
    sign_muon_step,
    muon_step,
    ns_dense_flops,
)

__all__ = [
    "bf16_rne", "fma_f32", "to_f32", "QUINTIC", "CUBIC", "momentum",
    "frobenius_normalise", "newton_schulz", "blockwise_newton_schulz", "sign_of", "pack_signs",
    "pack_signs_loop", "unpack_signs", "majority_vote", "int8_sum_vote", "post_vote_polar",
    "apply_update",
    "apply_update_f64", "sign_muon_step", "muon_step", "ns_dense_flops",
    "orthonormalise_columns", "column_normalize", "dion_step",
]
