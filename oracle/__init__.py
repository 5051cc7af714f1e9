"""Plain fp64 CPU oracle for absorbed-MLA latent decode.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import or run anything in this
package.  The product path (the CUDA library and its Python binding) never
imports it and shares no code, table or helper with it.

Contents
--------
``mla_ref``   RoPE, the naive (expanded K/V) MLA decode, the absorbed MLA decode,
              the one-shot causal forward used by the incremental-decode pin,
              the paged-cache writer (the stored values of a cache row) and the
              closed-form byte counters.
``e4m3``      The OCP FP8 E4M3 code book, an encoder (round to nearest even,
              saturating) and a decoder.

Every function cites the passage of the pages it follows.  The pages are four
web pages on DeepSeek Multi-head Latent Attention (MLA); citations use each
page's title and the section / equation / table on it:

* "DeepSeek MLA 吸收式缓存：真实权重执行与 FlashMLA 架构边界" (the absorb audit)
* "80 行 PyTorch 从零写 DeepSeek 的 MLA" (the 80-line PyTorch MLA post)
* "DeepSeek-V2-Lite 真实权重执行审计" (the V2-Lite trace)
* "G5 MLA KV 访存建模设计规格" (the G5 MLA KV memory-access spec)

Pins (what fixes this oracle other than itself) live in ``tests/test_oracle_*.py``.
Functions whose values no pin fixes are marked "parity unpinned" in their
docstring.
"""
