"""CPU oracle of the OasisKV lookahead sparse decode hot path.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously correct
restatement of what the pages on OasisKV say the hot path computes.  Only the
test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it; the library and its Python binding never do, and
nothing here imports them.

Sources, cited by page title and section:
  [XR] "OasisKV: Scaling In-Decode KV Cache Beyond HBM with Lookahead Sparse
       Prefetching" - paper review on xllm-io.github.io (Chinese).  Sections
       are numbered as on the page: §2 core idea (problem definition), §3
       architecture (Fig. 5, eqs. (1)-(4), the component table, the decode
       flow), §4 innovations (Figs. 4, 6, 7), §5 implementation, §6 experiments
       (Table 2 fetch-cap ablation, top-K sensitivity).
  [LX] the same title on lode.cx - summary article ("The Insight").
  [LP] "Scaling KV Cache Beyond Memory Limits" on legiblepapers.com - Key
       Takeaways, Summary & Methodology Analysis, FAQ Q1-Q9.
  [RP] researchpod.app episode page - abstract and transcript.

Modules:
  summary    per-block per-dimension min/max key summaries (Quest style)
  score      draft-query block scoring against the summaries
  select     per-KV-head top-K with capped eviction, transfer plan, table
  stage      host tile -> HBM slot copy named by the plan
  attention  sparse decode attention over the head-wise table (float64)
  sizing     eqs. (1)-(4) and the summary / KV byte counts
  pipeline   one layer of the whole path for a set of segments

Parity status: every function is pinned by the tests listed in its module
docstring.  One quantity of the pages is "parity unpinned": the agreement of
draft-query top-K with true-query top-K ([XR] §4, Figs. 4 and 6) needs real
models and is not computed here.
"""
