"""PolyKV CPU oracle -- TEST INFRASTRUCTURE, not part of the product.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its cpu_baseline
leg and its ``--impl reference`` arm) may import this package. The CUDA library
in ``serving_q8_encode_gb300`` never calls it and shares no code, header,
table or constant with it.

What it computes follows the PolyKV abstract ("PolyKV: A Shared
Asymmetrically-Compressed KV Cache Pool for Multi-Agent LLM Inference",
abstract): one compressed KV pool written once and read by N agents; keys as
int8 q8_0; values rotated by a Fast Walsh-Hadamard Transform and quantized
with a 3-bit Lloyd-Max codebook fitted to N(0,1).

Precision: the encode steps decide integers (codes), so they run in fp32 with
a fixed operation order that the GPU kernels also follow; attention runs in
float64 over the dequantized pool (the plain definition).

Parity status per function (what pins it is in tests/test_oracle_pins.py; each planted
mistake there -- an FWHT sign, half-even rounding, the pack bit order, the GQA head mapping --
turns a pin red):
  codebook.lloyd_max_normal     pinned (Max 1960 table, quadrature, sampled k-means)
  keys.quantize_q8_0            pinned (exact-rational brute force, round-trip bound)
  values.fwht_*                 pinned (scipy Hadamard matrix, self-inverse, norm)
  values.encode_values          pinned (nearest-centroid brute force, sum u^2 = d, NMSE)
  values.pack_codes             pinned (hand-packed 32-token group, round trip, group independence)
  attention.attend              pinned (closed forms: q=0 mean, T=1, dominant key,
                                constant V, two-token logistic, GQA mapping)
  accounting.*                  pinned (abstract's 2.91x, 97.7%, 0.45 GB)
  accounting: 19.8 GB absolute  parity unpinned (inconsistent with the model shape)
"""
from . import accounting, attention, codebook, keys, values  # noqa: F401
