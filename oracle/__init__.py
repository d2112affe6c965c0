"""Reference oracle for per-head-budget block-sparse attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import or run anything in this
package.  The CUDA library never calls it, and it shares no code with the
library (no kernels, headers, helpers or tables); the only shared module is the
seeded input generator in ``workloads``, which holds none of the method's
arithmetic.

Everything is plain, slow and written to be checked by eye against the pages:
floating point in fp64 (inputs are bfloat16 bit patterns promoted exactly),
integers in Python ints, exact sort-based top-k with ties to the lower block
index.

Sources (page title, then section):

* "S-HPLB: Efficient LLM Attention Serving via Sparsity-Aware Head Parallelism
  Load Balance" (Italian and Chinese summaries): offline profiling to a 90%
  attention-weight recovery ratio, Max-Min budget shifting with the total held
  fixed, and the greedy longest-first multiway partition (sort by budget,
  hand each item to the least-loaded worker).  Sections "Metodologia" A/B
  (Italian) and 2.1/2.2 (Chinese); the naive in-order assignment is in the
  Chinese summary's plain-language part, "第二招：负载均衡".
* "Riepilogo Tecnico: Fluxion": block-granularity top-k, the attention-sink
  block, and streaming vs retrieval heads ("Intuizioni Chiave" 1 and 2).
* "Unifying Sparse Attention with Hierarchical Memory for Scalable
  Long-Context LLM Serving" (Spin): the Index / Select / Attention split of the
  pipeline ("Abstracción de Partición Unificada").

Modules: ``plan`` (budgets and schedules), ``calib`` (coverage calibration to
demands), ``attention`` (pooling, scores, selection, sparse prefill attention),
``decode`` (the decode step), ``granularity`` (per-head block sizes and
budgets for decode retrieval heads).  Every function is pinned by CPU tests against
closed forms, brute force, or library routines (see ``tests/test_oracle_*``).
"""
