"""CPU oracle for the CSA2 decode path.  TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously-correct numpy code (float64 wherever the pages do not
fix a precision).  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import it.  It shares no code with the CUDA
library and imports nothing from it; both sides see the same seeded inputs
from ``synth``.

What each module follows:

* ``formats``   - FP4 E2M1 and FP8 E4M3 value sets and round-to-nearest-even
  encoders (the pages name the formats: trawling.dev "DeepSeek-V4.1-Flash
  공개", section "CSA2와 FP4 KV 캐싱"; origotech.dev deep dive, subsection
  "FP4와 SWA Bounded Replay"; the value sets are the public OCP definitions).
* ``append``    - RoPE then quantise-and-append of the main KV (FP4, one E4M3
  scale per 16 channels), the indexer key and the SWA KV (FP8).
* ``indexer``   - indexer scores, block scores, Full / Reindex / Reuse
  selection (origotech.dev deep dive, subsection "Compressed Sparse
  Attention 2(CSA2)").
* ``attention`` - one softmax over the selected global rows plus the window
  (ttj.kr article, section "CSA2와 어텐션 재설계").
* ``bruteforce`` - pure-Python loops for tiny inputs, used to pin the above.

Parity pins: every function here is pinned by ``tests/test_oracle_*.py``
against hand-derived worked examples, library routines (torch's float8
conversion, scaled_dot_product_attention) and brute force.  The page-level
byte budget (890 B/token) is not reproducible at these dimensions: parity
unpinned for that figure, and nothing here computes it.
"""
from . import formats, append, indexer, attention, bruteforce, pipeline  # noqa: F401
