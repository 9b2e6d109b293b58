"""CPU oracle for the Medusa decode step -- TEST INFRASTRUCTURE ONLY.

Plain, slow, fp64 numpy restatement of what one Medusa decode step computes,
written from the source pages and nothing else.  It shares no code with the
CUDA library and imports nothing from it.  Only the tests, the smoke check and
the benchmark's CPU-baseline leg may import this package; the library's product
path never does.

Sources (cited by page title and section):
  [ULT]  Ultralytics glossary "Medusa Heads": section "How the heads predict the
         next tokens" (head formula and its PyTorch example with the printed
         result [True, True, True]); section "Tree attention and accepting
         tokens" (2 x 3 Cartesian tree, ancestor-only mask, longest accepted
         branch, greedy match, typical acceptance).
  [WIB]  wiblog.cn "Medusa multi-head speculative decoding": sections
         "Medusa decoding heads", "Tree attention", "Typical acceptance",
         "Inference flow in an online chat service", "How the acceptance rate
         shapes the speedup".
  [CNN]  cnnetsun.cn "Medusa safety considerations": section "Posterior
         probability evaluation" (evaluate_posterior call and its outputs
         best_candidate, accept_length) and section "Key safety parameters"
         (posterior_threshold = 0.09, posterior_alpha = sqrt(threshold) = 0.3).
  [JIS]  jisaku.com glossary "Medusa (LLM decoding)": section "How Medusa works"
         (K heads, per-head top-k, tree of candidates, longest valid sequence).

Parity status: every function here is pinned by a `-m "not gpu"` test against
a fact the pages or mathematics fix (see tests/test_oracle_pins.py), except
where a function's docstring says "parity unpinned".
"""
from .medusa import (  # noqa: F401
    bf16_round, medusa_heads, tree_heads, head_topk, base_root,
    TreeTables, tree_tables, tree_tokens,
    apply_rope, tree_attention, verify_logits, node_posterior, nucleus_next, typical_accept, kv_commit,
    run_step, StepResult,
)
