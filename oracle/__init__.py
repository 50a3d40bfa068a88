"""CPU oracle for the OSCAR INT2 KV-cache serving path.

TEST INFRASTRUCTURE. This package is a plain, slow NumPy (float64) restatement
of what the serving path computes, written from the method's published
description. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import it; the product path never does, and it shares no
code, table or helper with the CUDA library.

Sources (cited by page title and section):
  [IT]  "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache
        Quantization", gist.science explainer (Italian), "Riepilogo Tecnico".
  [ES]  "Juntos, AI Open-Sources OSCAR: un sistema de cuantificación de caché KV
        de 2 bits consciente de la atención ..." (7minutos.es).
  [JA]  "技術概要：OSCAR - 2 ビット KV キャッシュ量子化のためのオフライン
        スペクトル共分散感知回転", gist.science explainer (Japanese).

Parity status per function (what pins it, see tests/test_oracle_*.py):
  hadamard ........................ pinned (scipy Sylvester matrix, Lemma 1)
  bit_reverse_index / matrix ...... pinned (textbook d=8 table, tier property)
  query_covariance ................ pinned (logit-error identity, closed form)
  score_weighted_value_covariance . pinned (brute-force double sum)
  eig_desc / composite_rotation ... pinned (orthogonality, Lemma 1 on R^T C R, key logit
                                    error below Hadamard-only when keys share the
                                    queries' leading directions)
  quantize_groups ................. pinned (brute force over all code vectors)
  layout codec .................... pinned (hand-worked byte fixture, round trip)
  decode_attention ................ pinned (torch SDPA float64, rotation equivalence)
  footprint_bits_per_element ...... pinned (the pages' 2.28 / 2.38 BPE, 8x, 0.24 %)
  clip_threshold .................. parity unpinned (the percentile reading is ours)
"""

from .oscar_oracle import (  # noqa: F401
    hadamard,
    bit_reverse_index,
    bit_reversal_matrix,
    query_covariance,
    causal_softmax_scores,
    score_weighted_value_covariance,
    eig_desc,
    composite_rotation,
    clip_threshold,
    calibrate,
    rotate,
    quantize_groups,
    dequantize_groups,
    cache_regions,
    next_state,
    OracleCache,
    decode_attention,
    logit_error,
    logit_error_from_covariance,
    footprint_bits_per_element,
)
from .layout_codec import (  # noqa: F401
    PAGE_BLOCK_BYTES,
    page_block_bytes,
    encode_page_block,
    decode_page_block,
    k_code_location,
    v_code_location,
    meta_location,
)
