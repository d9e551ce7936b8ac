"""fp64 CPU oracle for the speculative-decoding verify step.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` use it. It shares no code with
the CUDA library (``target_model_verify_gb300``) and imports nothing from it.

What it computes, and where the pages fix it:

* ``philox``   -- Philox4x32-10 (Salmon et al., SC'11, "Parallel random
  numbers: as easy as 1, 2, 3") and the two 24-bit uniform maps that drive
  the acceptance draw r and the residual/bonus draw u.
* ``verify``   -- the verify step: LM-head logits z = h W^T in fp64, p and q
  as softmax at temperature T, the acceptance rule and first-reject
  truncation, the residual / bonus sampler, and the greedy variant.
  "推测解码" (world.lapla.si/zh/specdec), sections 留下对的，换掉错的 and
  通过的规则; greedy: maxstudionews.com article 1664 (the verify paragraph)
  and "推测解码", section 先让小模型猜.
* ``tree``     -- tree verification: the same rule at every fork of a token
  tree (siblings in order, the residual renormalised after each rejection),
  "推测解码", section 不要第二个模型; a chain-shaped tree is the chain step.
* ``attention`` -- verify-step attention: the gamma + 1 new positions of a
  sequence over its KV cache, causal among themselves, grouped-query heads
  ("推测解码", section 几段话一起写: every sequence reads its own cache).
* ``cluster_head`` -- the drafter's clustered LM head: cluster logits, the
  top-k clusters, token logits of their members only, the draft token
  ("多詞元預測視覺化指南", section 高效嵌入器).
* ``formulas`` -- the closed forms the same page prints: tokens per weight
  read, speedup, arithmetic overhead (sections 接受率 α, 快多少,
  用的是闲着的算术).

Pins (tests/test_oracle_pins.py, tests/test_oracle_tree_pins.py,
tests/test_oracle_attention_pins.py, tests/test_oracle_cluster_pins.py) tie
every
function to something other than itself: a library Philox (triton's
interpreter), brute-force loops, exact enumeration over all 2^24 uniform
values, exact rational enumeration of the tree rule's output law, chi-square
and binomial bounds, and the numbers the page prints. No function here is
"parity unpinned".
"""
