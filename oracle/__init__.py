"""Plain, slow CPU oracle for the routed-expert cache hot path.

TEST INFRASTRUCTURE, NOT PRODUCT CODE. Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference arm of ``bench.py`` may import anything here.
The CUDA library never routes through this package, and this package imports
nothing from the CUDA side (``expert_cache_gb300``).

Pages cited (by title; sections as printed on each page):

  [EXPLAINER] "FreeToken: Efficient Edge-Native MoE Serving with Bandwidth-Adaptive
              Execution" (jjl357.github.io blog explainer of the arXiv v1 paper)
  [QIITA]     "FreeTokenってなんだ？ ─ 8GBノートPCで35Bを動かす判断基準" (Qiita)
  [BWRATIO]   "FreeToken hybrid MoE 后端：带宽比如何决定专家「搬」还是「算」"
              (wanger-sjtu.github.io source walkthrough)
  [JUHE]      the juhe.plus article on running Qwen3.6-35B-A3B on an 8 GB
              RTX 4060 Laptop with FreeToken (untitled feed page; cited by its
              section headings)

Modules:
  formats          E2M1 / E4M3 codecs, NVFP4 weight and activation quantisers,
                   the per-flat-id expert record
  qrule            the integer q* split rule and the bandwidth -> Q16 fraction forms
  lru              the global cross-layer LRU slot cache (OrderedDict) and a
                   brute-force history-based twin
  moe              dense fp64 MoE-layer definitions for decode and prefill
  static_placement the static (prefill-time) placement baseline simulator

Parity status: every function here is pinned by a ``-m "not gpu"`` test against
what the pages or the mathematics fix (see ``tests/test_oracle_*.py``); none is
"parity unpinned".
"""
