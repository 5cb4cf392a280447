"""CPU fp64 oracle for the 3-D tensor-parallel layer cube.

TEST INFRASTRUCTURE ONLY.  This package is the plain, slow, obviously
correct statement of what the GPU path computes.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it.  The product package never imports it, and it shares no code,
header, table or helper with the product; both sides only share the seeded
input generators in ``synth_inputs.py``, which hold none of the method's
arithmetic.

Sources (cited by page title and section):

* "Maximizing Parallelism in Distributed Training for Huge Neural Networks"
  (Bian, Xu, Wang, You; arXiv 2105.14450), written MP3D below:
  §2.3 (3-D parallel matrix multiplication), §3.1.1 (Load Balancing),
  §3.1.2 (Matrix-matrix operations, Algorithms 1-6), §3.1.3
  (Matrix-vector operations, Algorithms 7-8), §3.2 (Parallel Transformer
  layers).
* "On Optimizing the Communication of Model Parallelism" (arXiv 2211.05322),
  written CMR below: §2 (device mesh, sharding spec, data slice, cross-mesh
  resharding and unit communication tasks, Figure 2).
* "Transformer Training 11: Model Parallelism" (lecture deck), written TT11
  below: section "Tensor parallelism" (column-split FFN with local GELU,
  row-split second matrix with summed partials).

Modules:

* ``layouts``  - the cube layouts, the diagonal vector layout, the
  mesh sharding specs, sharded storage, resharding and unit tasks.
* ``linear``   - the 3-D linear (C = A.B [+ b] [GELU]) and its gradients.
* ``mlp``      - the Megatron / cube MLP.
* ``layer``    - the pre-LN GPT decoder layer, forward and backward.
* ``metrics``  - the error metric the parity tests use.

Parity status per function is stated in each module header.
"""
