"""Plain, slow, float64 CPU oracle for tiled exact attention ("Flash MSA").

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` use it.  It shares no code with
the CUDA library (``tiled_exact_attention_flash_gb300``) and never imports it;
both sides receive the same seeded inputs from
``tiled_exact_attention_flash_gb300.inputs``, which holds none of the method's
arithmetic.

What it computes (one attention head at a time, float64 throughout):

* ``mask.live_matrix`` -- the element predicate of the mask: causal, local
  window +-W, block dilation, fixed strided key blocks ("How Does Flash-MSA
  Sparse Attention Work", section "How Flash-MSA Sparse Attention Works",
  the list of mask kinds; causal from "Flash MSA Attention Kernel
  Implementation", section "Optimization Tricks That Actually Matter",
  paragraph "Masking and causal attention").
* ``attention.forward_head`` / ``attention.backward_head`` -- the plain
  definition O = softmax(mask(Q K^T * scale)) V with masked scores set to
  -inf, LSE = log-sum-exp of the live scores, and the analytic gradients
  ("Flash MSA Attention Kernel Implementation", sections "Why Standard
  Attention Broke" and "The Backward Pass: The Real Beast").
* ``loops`` -- a scalar triple-loop restatement (tiny N) and a tiled
  online-softmax restatement ("Flash MSA Attention Kernel Implementation",
  section "The Flash Core: Tiling Over the Memory Hierarchy").
* ``block_index`` -- classification of every 128 x 128 tile as dead / full /
  partial by evaluating the element predicate on all of its entries, and the
  CSR / CSC / longest-row-first orders built from it ("How Does Flash-MSA
  Sparse Attention Work", the precomputed per-block index list); packed
  variable-length sequences with causal / window masks are tiled per
  sequence (``sequence_tiles``), each from its own first token.

Pins (``tests/test_oracle_pins.py``, run with ``-m "not gpu"``): uniform
attention for Q = 0, causal row 0, one-hot dominant rows, constant V, row sums
of P, gradient-sum invariants, permutation invariance, central finite
differences, agreement with the scalar loops and with the tiled online-softmax
restatement, closed-form live-tile counts for the benchmark masks, the
per-sequence tiling equal to every sequence's own index, and
negative controls (mistakes planted in copies of these functions must fail a
pin).  Every function here is pinned; none is "parity unpinned".
"""
