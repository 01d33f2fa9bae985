"""Float64 CPU oracle for tiled-online-softmax attention -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU baseline
leg and its ``--impl reference`` arm) may import this package.  The library in
``attention_attn_prefill_gb300`` never imports, links or runs it, and this
package never imports the library: the two share no code.  Inputs come from
``workloads`` (random numbers only).

Modules:
  attention  -- the exact definition in float64 (prefill, paged decode, the
                split/combine decomposition); every function is pinned by tests.
  numerics   -- float32 / bfloat16 rounding helpers (round to nearest even).
  split_sim  -- the scalar group-split simulations of the long-context decode
                page: the group geometries, per-group rounding and merges of
                the Triton, FlashAttention-2, XQA and TensorRT-LLM decode
                algorithms, under float32 or exact arithmetic, and the
                FlashAttention-2 split-count heuristic.

Parity status: every function here is pinned by closed forms, invariants,
brute force on tiny inputs or values the pages print (see tests/).
"""
