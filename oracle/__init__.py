"""fp64 CPU oracle for the DSpark per-step path — TEST INFRASTRUCTURE ONLY.

This package is the plain, slow, obviously correct reference that the CUDA
library is checked against.  Only `tests/`, `__graft_entry__.smoke()` and the
CPU-baseline / reference legs of `bench.py` may import it.  The product path
(the C-ABI library and its Python binding) never imports, links or executes
anything here, and nothing here imports the product path.

Sources cited in this package (page titles; sections named on each page):

* [DSpark] "DSpark: Confidence-Scheduled Speculative Decoding with
  Semi-Autoregressive Generation" (papercache.org summary of the paper).
* [MTP Survey] "大模型推理 MTP 算法 Survey" (backyes.github.io).
* [DeepSpec analysis] the bevisy.github.io page on speculative decoding and the
  DeepSpec project.
* [Random123] Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
  1, 2, 3", SC'11 — the Philox4x32-10 generator (the pages name no RNG; the
  counter-based Philox contract is this library's own choice).

Modules:
  philox    Philox4x32-10 and the (seed, request, position, draw) uniforms
  sampling  inverse-CDF sampling with fp64 margins
  draft     Markov-head draft sampler + confidence head
  schedule  Sequential Temperature Scaling, Algorithm 1, flatten + markers
  verify    lossless rejection-sampling verification

Every function computes in fp64 unless its docstring says otherwise (the
scheduler's survival products are fp32 by contract, because they are sort keys
that both sides must reproduce bit for bit).
"""
from . import philox, sampling, draft, schedule, verify  # noqa: F401
