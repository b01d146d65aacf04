"""Plain fp64 CPU oracle for the OSCAR-style rotated INT2 KV-cache hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute anything in this package: only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.
It shares no code, table or constant generator with the CUDA library
(``rotated_int2_kv_gb300``); the two meet only in the seeded synthetic inputs
that tests hand to both.

Sources (web pages, cited by title and section):

* [OSCAR news] "Together AI、OSCARをオープンソース化：長コンテキストLLMサービング
  のためのアテンション認識2ビットKVキャッシュ量子化システム" (news article on
  OSCAR, Offline Spectral Covariance-Aware Rotation).  Sections used:
  "OSCARの違い" (logit-error identity, C_Q, C_S, R = U·H·P_br) and
  "サービングシステム：混合精度キャッシュレイアウト" (64 BF16 sink tokens,
  256 BF16 recent tokens, INT2 history after rotation and clipping).
* [Escha log] "RTX 5070×2(12GB×2)でQwen3.8-27B-Escha-W2を動かす" (deployment
  log), part 2 "KVキャッシュも2bitにして長コンテキストにする": fix 1 (0.25 byte
  per element), fix 3 (Sylvester Hadamard / sqrt(head_dim), exact
  orthogonality in fp32), fix 4 (query head -> KV head mapping), the
  "--kv-cache-quant-group-size 64" settings table, and the supplementary
  table of INT2 KV bytes per token.
* [Scheduler log] "12GB の VRAM に 27B" scheduler article: page_size 1
  (token-granular page table).
* [Prefix log] "KVプールが上限だった — hybrid GDN の長文キャッシュ…": the INT2
  prefill path expands the cached prefix to fp16 in a workspace
  (dequantize_prefix_kv) before attention.

Modules:
  rotation   -- Hadamard, bit reversal, eigenbasis, R = U·H·P_br, covariances
  quant      -- bf16 and E4M3 rounding, clipped group-wise asymmetric INT2
                quantiser (fp16 or E4M3 scale and zero), 2-bit packing,
                record and slot serialisation
  cache      -- the three-region cache and its append semantics
  attention  -- exact-softmax decode attention over the mixed cache, and the
                split/LSE merge
  prefill    -- exact-softmax attention of a prefill chunk over the cached
                prefix and its own keys (causal)
  accounting -- bytes and bits per token / element
"""

from .rotation import (hadamard, block_hadamard, bitrev_indices, eig_desc, build_rotation,
                       covariance, value_covariance)
from .quant import (bf16_round, e4m3_round, quantize_rows, dequantize_rows, pack_codes,
                    unpack_codes)
from .cache import OracleConfig, OracleCache, regions
from .attention import decode_attention, decode_attention_split
from .prefill import prefill_attention
from .accounting import (code_bytes_per_token, record_bytes, bits_per_element,
                         window_fraction)

__all__ = [
    "hadamard", "block_hadamard", "bitrev_indices", "eig_desc", "build_rotation", "covariance",
    "value_covariance", "bf16_round", "e4m3_round", "quantize_rows", "dequantize_rows",
    "pack_codes", "unpack_codes", "OracleConfig", "OracleCache", "regions",
    "decode_attention", "decode_attention_split", "prefill_attention", "code_bytes_per_token",
    "record_bytes", "bits_per_element", "window_fraction",
]
