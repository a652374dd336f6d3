"""CPU oracle for the paged KV store hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (the CUDA library and its Python binding) never
imports, links or executes anything here, and this package imports nothing
from the product.

Everything is plain NumPy in float64, written from the "Paged KV cache"
maintainer design page of the NInfer engine (the typed growing KV pool
contract) and from this library's stated codec rules:

* ``formats``   – exact scalar number formats (fp16, E4M3FN, E2M1) with
                  round-to-nearest-even; pinned against numpy's float16 cast
                  and an exhaustive nearest-value search.
* ``codec``     – the five KV profiles: BF16, INT8-G64, FP8-E4M3FN-row256,
                  NVFP4-G16 and the asymmetric K8V4.
* ``layout``    – plane schema, page-major / head-major address formulas,
                  per-token byte table, capacity bounds M_min / M_max.
* ``store``     – a byte image of a pool: paged append, gather through block
                  tables, partial-tail copy-on-write.
* ``attention`` – causal GQA softmax attention (decode / verify / chunked
                  prefill) in float64, with the natural-log LSE.

Parity status of each function is stated in its module docstring.
"""

from . import formats, codec, layout, store, attention  # noqa: F401
