"""CPU oracle for exact scaled-dot-product attention (TEST INFRASTRUCTURE ONLY).

This package is the plain, slow, obviously correct statement of what the GPU
path computes.  Only the tests, the smoke check and the benchmark's CPU
baseline may import it; the library and its Python binding never do, and the
two share no code.

Pages cited (by title and section):

* [ZeRO-vs-FA]  "ZeRO 与 FlashAttention 各优化什么?" -- sections
  "注意力瓶颈与优化路线" and "FlashAttention 与 ZeRO 必须分开" (the method is
  exact dense attention, only HBM traffic changes).
* [FA-memory]   "38.解释FlashAttention的显存优化原理" -- part 1 (the N x N
  score/softmax matrices), 2(1) tiling with 128-token blocks, 2(2)
  recomputation in the backward pass.
* [QBank-36]    "十九、分布式与系统方向的标准答案速查区", question #36
  "FlashAttention 为什么常被说成是 IO-aware（面向 IO 的）优化？" -- part 2
  (standard attention S = QK^T, P = softmax(S), O = PV over B x H x L x d
  tensors), part 3 (tiling + online softmax), part 7 (backward recompute).
* [Lecture]     Stanford lecture summary (youtublog.net) -- sections
  "GPU 显存和注意力瓶颈" (causal self-attention), "推导 FlashAttention 的在线
  softmax" (running max, numerator/denominator, rescale by exp(old-new)) and
  "减少缓存表示并验证草稿" (grouped-query attention with G key/value groups).

Modules:

* ``ref``   -- NumPy fp64 definition (row-blocked, full rows of S and P).
* ``brute`` -- the same definition in pure-Python loops, for tiny shapes.
* ``online`` -- the pages' streaming numerator/denominator recurrence, used
  only to pin the definition against the pages' own derivation.

Parity status: every function here is pinned by tests under ``tests/`` that
do not call back into the same arithmetic (closed forms, brute force, finite
differences, library routines, the three-element worked example).
"""
