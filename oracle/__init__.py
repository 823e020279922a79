"""CPU oracle for the FlashOverlap signaled-GEMM + reorder path.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference legs of ``bench.py`` use it.  It shares no code, table or constant
with the CUDA path under ``communication_overlap_gb300/``.

It is a plain, slow restatement of what the path computes, written from two
web pages:

* [P1] "FlashOverlap: 信号驱动计算通信重叠论文详解" (a deep-dive of
  arXiv:2504.19519), sections 一、信号机制, 二、重排机制, 三、Wave Group
  划分设计空间.
* [P2] "Efficient and Adaptable Overlapping for Computation and
  Communication via Signaling and Reordering" (abstract and the captions of
  Figures 3 and 5).

Modules:
  bf16    -- IEEE round-to-nearest-even to bfloat16, from the format's definition
  plan    -- tile order, waves, wave groups, counting table, mapping tables, layouts
  gemm    -- fp64-accumulated GEMM rounded once to bf16
  comm    -- pre-comm reorder, the four communication stand-ins, post-comm reorder
  pipeline-- one whole pass of the path (used by tests and the CPU baseline)

Where the pages leave a step open, the function that takes the step states
the reading it uses in its own docstring.
"""
