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

Modules (and the CPU tests that pin them)
-----------------------------------------
encoders   fp32 -> bf16 / fp16 / e4m3 bit encoders written from the format definitions
           (test_oracle_encoders)
philox     Philox4x32-10 counter-based generator and the dither stream (test_oracle_philox)
quant      quantize-on-append for every layout (INT8 with one scale per token, per 32-channel
           group, or with the fixed-channel outlier bypass), dequantization, band-norm and value
           witnesses (test_oracle_quant, test_oracle_groups, test_oracle_bypass, test_oracle_value)
attention  exact and compressed attention, total variation, Tier A / Tier B meter, value side,
           alternative bound shapes (test_oracle_attention, test_oracle_groups, test_oracle_bypass,
           test_oracle_value, test_oracle_shapes)
meter      meter finalisation, coverage, per-request risk ranking, gate contributions and the
           greedy page-in plan (test_oracle_meter_bytes, test_oracle_gate)
bytes      byte account per layout and per workload (test_oracle_meter_bytes, test_oracle_groups)
rope       binary32 RoPE-on-append and its cos/sin table (test_oracle_rope)

Parity status: every function here is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_*.py``; the Philox generator is additionally pinned word for
word to the CUDA toolkit's own Philox4x32-10 by a GPU test (see
``oracle/philox.py``).
"""
