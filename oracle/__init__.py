"""fp64 CPU oracle for round-robin sequence-shard DSA prefill attention.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or execute this
package; only `tests/`, `__graft_entry__.smoke()` and `bench.py`'s CPU-baseline leg do.
It shares no code with the CUDA path (`deepseek_v3_sparse_round_gb300/`), and that path
never imports it.

One module per step, each written from its defining passage:

  split.py    round-robin split: shard token list, batch ids, positions, shard cu_seqlens
              ("[DeepSeek v3.2] 上下文并行详解", section 2.B and section 4 part 3 step 1)
  rerange.py  all-gather layout and rerange to logical order (same page, section 2.C and
              section 4 part 3 step B)
  inseq.py    contiguous in-seq-split comparator (same page, section 4 part 1)
  indexer.py  lightning-indexer scores I[t,s] = sum_h w[t,h] ReLU(q_idx[t,h] . k_idx[s])
              over the causal history (the DeepSeek-V3.2 DSA lightning indexer; the pages name
              it the bottleneck: "[RFC]: Parallel strategy for Deepseek v3.2 like models")
  topk.py     per-query top-k by a full stable sort, lowest index wins ties
  mla.py      sparse MLA over the selected latent rows, and dense causal MLA

All floating point is fp64, computed from exactly the values the GPU receives (bf16 inputs
widened). Every function is pinned by `tests/test_oracle_*.py` against worked examples,
closed forms, brute force on tiny inputs and invariants.
"""
