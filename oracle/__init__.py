"""CPU oracle for the DTensor tensor-parallel linear and its layout transforms.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library,
its C ABI or the Python binding) imports, calls or links this package.  Only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it.

The oracle is written to be checked by eye against the pages it follows, not
to be fast.  It shares no code with the CUDA path: it has its own bf16
rounding, its own placement arithmetic and its own sums.  Every function
cites the passage it restates.  Sources (by page title and section):

* "DTorch user guide -- Module parallel" (tingkuanpei.github.io/dtorch, the
  Chinese and English editions): section 3, "Linear implementation
  walkthrough" -- weight/bias placements per ``tp_shard_type`` and the
  input/output placement checks.
* "Hyper-Parallel DTensor API" (MindSpore hyper-parallel pull request 121):
  ``distribute_tensor`` (with printed per-rank values), ``redistribute``,
  ``reduce_partial``, ``full_tensor``, the ``shape`` property and the
  placement-type table.
* "Model parallelism" (wineandchord.com, LLM systems): "Tensor Parallel"
  (column- and row-parallel equations) and "Tensor-parallel linear layers"
  (the single-process reference with ``torch.chunk`` shards, the worked
  example x[3,8] @ W[8,12] with 4 parts, and the coverage invariant).
* "nanotron tutorial, chapter 5: 3D parallelism" (jwzheng96.github.io):
  section 5.1 (TensorParallelColumnLinear / RowLinear, ALL_REDUCE and
  REDUCE_SCATTER modes) and section 5.5 (mode choice).

Modules
-------
bf16        IEEE binary16-brain rounding and widening (numpy bit patterns).
placement   Mesh coordinates, torch.chunk-style block split, slots and boxes.
redistribute  Global assembly (in-order fp32 Partial sums) and slicing.
linear      fp64 column/row parallel linears, TP MLP, attention projections.
embedding   EmbeddingWithReplicateOutput gather.

Parity status: every function here is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_*.py``; the readings the pages leave open are listed in
the repository's design notes.
"""
