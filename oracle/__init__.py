"""Plain, slow CPU oracle for the paged KV cache and PagedAttention decode.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute anything in this package: only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` use it.  It shares no code, header,
table or helper with the CUDA library in ``paged_kv_cache_295_gb300``, and
imports nothing from it.

Modules (each function cites the passage of the source pages it follows; the
pages are "LLM inference tutorial" (xurj.top, Tutorial/Detail/167), "nano-vLLM
architecture" (intelliparadigm 2014318), "TGI architecture" (intelliparadigm
2004249) and "ToPG framework" (intelliparadigm 2232463)):

* ``pool``      - FIFO physical-block pool, per-block refcounts, per-sequence
                  block tables and slot arithmetic ("LLM inference tutorial",
                  section 4.2 PagedKVCache and 4.3 Prefix Caching; "nano-vLLM",
                  section 4.3 memory-pool formula).
* ``fp8``       - OCP FP8 E4M3 decode / round-to-nearest-even saturating encode,
                  written from the format definition.
* ``attention`` - the append (cache write by slot) and decode attention as the
                  plain definition: gather the sequence's blocks into
                  contiguous K/V, then softmax(q K^T * scale) V in float64
                  ("LLM inference tutorial", sections 4.1, 4.2 get_kv, 4.4
                  MHA/GQA/MQA forward).
* ``prefill``   - paged (chunked) prefill attention: a chunk of query tokens,
                  the last positions of their context, attends causally over
                  the gathered cache ("LLM inference tutorial", sections 1.2
                  prefill phase, 4.4 forward, 6.2 chunked prefill).

Every float computation here is float64 unless a step is defined by a narrower
type (FP8 dequantisation is one float32 multiply, as stated in ``attention``).
"""
