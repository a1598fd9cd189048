"""Oracle for the Sarathi hybrid-batch decoder step -- TEST INFRASTRUCTURE ONLY.

A plain, slow, CPU restatement (NumPy, float64 unless a caller asks for
float32) of what the hybrid-batch step computes, written from the pages that
describe the method, never from the CUDA library.  Only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference leg of
``bench.py`` may import it.  The product path (``chunked_prefill_hybrid_sar_gb300``)
never imports it and shares no code with it; the only common module is
``synth`` (seeded input draws).

Page titles cited in this package:

* "SARATHI技术：大模型推理优化的分块预填充与混合调度" -- the engineer's write-up
  (cited as *SARATHI technique write-up*).
* "SARATHI: Efficient LLM Inference by Piggybacking Decodes with Chunked
  Prefills" reading notes (cited as *SARATHI reading notes*).
* "Taming Throughput-Latency Tradeoff in LLM Inference with Sarathi-Serve"
  paper digest (cited as *Sarathi-Serve digest*).
* the Sarathi-Serve project overview article (cited as *Sarathi-Serve overview*).

Modules:

* ``model``  -- decoder layer, chunked prefill, hybrid stacked step.
* ``sched``  -- stall-free batching (Algorithm 3) and the page allocator.
* ``cost``   -- roofline time, tile count, batch-size bound, KV re-read count.

Parity pins: every function here is pinned by a ``-m "not gpu"`` test against
something other than itself (closed forms, library special cases, brute
force, the pages' printed numbers).  The absolute hidden-state values of a
random-initialised model have no printed worked example: beyond those pins
they are "parity unpinned".
"""
