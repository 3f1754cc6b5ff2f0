"""Oracle: a plain, slow, float64 CPU statement of what the quantized-KV decode path computes.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA library never calls it, and it never calls the CUDA library:
the two share no code.  Every function cites the passage of the source pages it
follows:

* "WitCert: Sound Runtime Risk Observability and Gating for KV-Cache
  Quantization" (arXiv 2607.28699) -- the meter (Tier A witness bound, Tier B
  dither certificate), the dithered INT8 quantizer and the split-KV merge.
* "Compress the shared cartridge. Keep the keys." (knlp.io, cartridge
  asymmetric quantization) -- the K16/V8 and K8/V8 layouts, the byte table and
  the shared-prefix single-softmax decode.

Modules
-------
encoders   fp32 -> bf16 / fp16 / e4m3 bit encoders written from the format definitions
philox     Philox4x32-10 counter-based generator and the dither stream
quant      quantize-on-append for every layout, dequantization, band-norm witness
attention  exact and compressed attention, total variation, Tier A / Tier B meter
meter      meter finalisation, coverage and per-request risk ranking
bytes      byte account per layout and per workload

Parity status: every function here is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_*.py``; the Philox generator is additionally pinned word for
word to the CUDA toolkit's own Philox4x32-10 by a GPU test (see
``oracle/philox.py``).
"""
