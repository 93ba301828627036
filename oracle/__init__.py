"""fp64 CPU oracle for position-independent KV stitching.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference arm of
``bench.py`` may import this package.  The library under
``position_independent_kv_stitch_gb300`` never imports it, shares no code
with it and must fail loudly (never fall back here) when its CUDA library is
missing.

What it computes is the plain definition of the method, in float64, written
from three pages:

* "EPIC Guide: Position-Independent Caching for LLM Serving" (aifetchly blog,
  on EPIC, ICML 2025) -- the RoPE rotation, the in-place shift
  ``k_target = R(dp) k_cached``, values untouched, the chunk registry and
  prompt composer, LegoLink's per-chunk sink tokens.
* "Irminsul: MLA-Native Position-Independent Caching for Agentic LLM
  Serving" (gist.science explainer) -- the MLA row (512-d latent copied,
  64-d rope key delta-rotated), ``delta = p_target - p_source``, the
  first-chunk carve-out of 32 tokens.
* "SemPIC: Learning Semantic Position-Independent KV Caches" (agihunt
  summary) -- cache-hit serving = assign final positions, re-rotate keys.

Pin status of each function (what outside fact each is checked against is in
``tests/test_oracle_*.py``):

* ``rope_inv_freq``      pinned (closed forms: base 2^d gives 2^-2i exactly)
* ``rotate``             pinned (identity, quarter-turn closed forms,
                         complex-product and rotate-half forward RoPE,
                         composition brute force, norms, relative position)
* ``llama3_inv_freq``    pinned by values derived by hand from the public
                         Llama-3.1 rule (not on the pages): blend weights of
                         exactly 1/4, 1/2 and 3/4, both regime edges, the
                         outer regimes, factor 1, and the regimes of
                         Llama-3.1-8B's own table.
* ``compose``            pinned (offsets printed on the EPIC guide's figures
                         and client request)
* ``BlockPool``          pinned (brute force on tiny requests)
* ``recompute_positions`` pinned (the EPIC listing's sink rule, the Irminsul
                         carve-out)
* ``stitch_*`` / ``rerotate_inplace`` pinned end to end against forward RoPE
                         computed at the target position.
* ``attention_decode`` pinned (uniform scores give the mean value, a dominant
                         score picks its value, token order does not matter,
                         shifting query and keys together changes nothing)
* ``sink_bias``          pinned (the EPIC listing's boundary loop)
* ``map_request`` / ``apply_mapped`` (virtual block mapping) pinned against the
                         block ids printed on the EPIC runtime figure and
                         against forward RoPE at the mapped positions.
* ``gear_hashes``        pinned (the explicit 64-token window sum, the closed
                         form of a constant stream, the window length itself)
* ``cdc_chunk_ends``     pinned (cuts exactly where the hash is below the
                         threshold; boundaries follow content when a prefix
                         shifts a document; min/max length invariants)
* ``xxh64``              pinned against the system xxHash library (libxxhash)
                         when it is installed
* ``s1_windows``         pinned (brute force)
"""

from .cdc_oracle import (  # noqa: F401
    GEAR_WINDOW,
    S1_WINDOW,
    gear_hashes,
    gear_hashes_window,
    cdc_chunk_ends,
    threshold_for_mean,
    xxh64,
    fingerprint,
    registry_key,
    s1_windows,
    chunk_document,
)
from .pic_oracle import (  # noqa: F401
    NEOX_HALF,
    INTERLEAVED,
    BF16_SENTINEL,
    Chunk,
    Segment,
    BlockPool,
    bf16_bits_to_f64,
    rope_inv_freq,
    llama3_inv_freq,
    model_inv_freq,
    rope_pairs,
    rotate,
    rotate_rows,
    compose,
    blocks_needed,
    recompute_positions,
    recompute_csr,
    stitch_paged,
    rerotate_inplace,
    expected_row,
    BlockChunk,
    MappedSegment,
    BusyError,
    map_request,
    release_request,
    apply_mapped,
    attention_decode,
    sink_bias,
)
