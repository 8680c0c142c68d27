"""fp64 CPU oracle for causal grouped-query attention against a KV cache.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` import this package. It shares no code with
the CUDA library and imports nothing from it.

Two independent formulations live here:

* ``oracle.core``  -- plain loops in C (``gqa_oracle.c``), fp64, the definition
  written out row by row; fast enough for sampled checks of full-size inputs.
* ``oracle.dense`` -- the explicit mask-matrix form of kopitiam-runtime
  src/attention.rs (``causal_mask``, ``repeat_kv_heads``, dense softmax) in
  numpy fp64, for tiny inputs. The tests hold the two to 1e-12 of each other.
"""
