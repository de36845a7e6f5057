"""CPU oracle for the compressed KV-cache hot path.  TEST INFRASTRUCTURE.

This package is the plain, slow, obviously-correct statement of what the
GPU path computes.  Only the test suite, the smoke check in
``__graft_entry__.smoke()`` and the CPU-baseline / reference arm of
``bench.py`` may import it.  The product (the ``bit_kv_cache_quant_gb300``
package and its CUDA library) never imports, links or runs anything here,
and nothing here imports the product: the two share only the seeded input
generator in ``synth``.

Sources (cited by page title and section throughout):

* "StreamingLLM + KIVI -- long-context decode without growing the KV cache"
  (tinygpt docs): sink + window middle eviction, the KIVI affine quantiser,
  the KIVI storage layout, the failure taxonomy.
* "SnapKV -- Prefill Observation-Window Token Eviction" (veloxquant-mlx
  docs): observation-window scoring, sink-forced top-k, keep-set storage.
* "kv-cache: optional per-channel K-cache mean-centering for Q4_0"
  (llama.cpp PR #51): symmetric Q4_0 K cache, per-(kv-head, channel) bias.
* "Low-bit KV caches on MLX: what exists and what is missing": per-token
  group-64 affine quantisation, bits-per-element arithmetic.

Precision: quantiser decisions (scales, zeros, codes) are taken in IEEE
fp32 with round-to-nearest-even, exactly as the kernels take them; stored
metadata is rounded to fp16; attention and SnapKV scores are float64.

Every function is pinned by ``tests/test_oracle_quantize.py``,
``tests/test_oracle_cache.py`` and ``tests/test_oracle_attention_snapkv.py``
against closed forms, brute force, special cases that reduce to library routines and the
pages' printed numbers (``tests/golden/``).  No function here is "parity
unpinned".  ``tests/test_oracle_mutations.py`` checks the pins in turn: each
of its cases plants one plausible slip in a function here (on the CPU, for
that case only) and requires a pin to fail.
"""
from . import quantize, cache, attention, snapkv, accounting  # noqa: F401
