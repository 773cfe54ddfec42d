"""CPU oracle for TurboQuant-style KV-cache compression (TEST INFRASTRUCTURE ONLY).

This package is a plain, slow, obviously-correct restatement of what the
compressed-KV hot path computes, written in numpy (fp64 unless a step is
defined in fp32).  It exists to check the CUDA library against.  Only the test
suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference
arm may import it; the product path (``compressed_attention_gb300``) never
does, and this package never imports the product path.  The two share no code;
the only common dependency is ``synth`` (seeded synthetic inputs, which holds
none of the method's arithmetic).

Sources and how they are cited
------------------------------
Every function names the passage it follows, by page and section:

* [turbo4 post-mortem] -- "turboquant_plus: how the turbo4 KV format came back"
  (hncyxsy.com/news/190332), sections 1-10 (1 starting point, 2 seven bugs,
  3 QJL ablation, 4 speed investigation, 5 4-bit breakthrough, 6 journey,
  7 validation, 8 lessons, 9 status and centroid investigation,
  10 independent verification).
* [Triton deep dive] -- "TurboQuant fused Triton kernels deep dive: 3 tricks for
  computing attention directly on the compressed KV" (0539edu.com/news/5502052),
  sections "why decode stalls on KV read-back", "trick 1: rotate the query
  once", "trick 2: precomputed query sketch", "trick 3: single-pass online
  softmax", "how the three kernels form one decode", "write path and codebook".
* [PolarQuant-KV] -- "PolarQuant-KV: dual KV-cache compression for consumer
  GPUs" (gsyq.cn/news/1549986), sections 2.1-2.3, 3.1-3.3.  Low reliability;
  used only for test ideas (distribution of rotated coordinates).

Readings of points the pages leave open are stated where they are used, in
the docstring of the function that takes them.

Parity status
-------------
Every function here is pinned by a ``-m "not gpu"`` test against something
other than itself (printed values, closed forms, textbook tables, brute force,
invariants), except the two stated below:

* "parity unpinned": the exact bits of the seeded dense rotation Pi and the QJL
  matrix S (the pages fix only "QR of a Gaussian" and "a Gaussian", not a
  generator); their distributional and orthogonality properties are pinned.
* "parity unpinned": the choice of the 8-level (turbo3) and 4-level (prod)
  tables as converged Lloyd-Max codebooks; they are pinned to their own
  fixed-point property and to Max's published Gaussian quantizer, not to a
  printed table for d=128.
"""

from .codebook import (  # noqa: F401
    make_codebook,
    quantile_codebook,
    lloyd_codebook,
    sphere_codebook,
    sphere_mass,
    stored_codebook,
    codebook_mse,
)
from .rotation import (  # noqa: F401
    splitmix64,
    wht_signs,
    fwht,
    wht_rotate_fp32,
    wht_rotation_matrix,
    gaussian_matrix,
    dense_rotation,
    qjl_matrix,
)
from .formats import (  # noqa: F401
    ROW_BYTES,
    canonical_norm_fp32,
    encode_turbo,
    pack_turbo4,
    pack_turbo4_rows,
    unpack_turbo4,
    unpack_turbo4_rows,
    pack_turbo3,
    unpack_turbo3,
    encode_prod,
    qjl_sign_bits,
    qjl_residual_estimate,
    pack_prod,
    unpack_prod,
    encode_vgroup,
    pack_vgroup,
    unpack_vgroup,
    Rotation,
    Codec,
)
from .attention import (  # noqa: F401
    gqa_kv_head,
    attention_reference,
    prefill_reference,
    attention_compressed_domain,
    online_softmax_merge,
)
