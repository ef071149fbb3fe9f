"""CPU oracle for the structured-slot-read denoise step (float64, NumPy).

TEST INFRASTRUCTURE ONLY.  This package is the plain, slow, obviously correct
statement of what the GPU path computes.  Only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
it.  It shares no code with the CUDA library (no kernels, headers, helpers,
tables or pre/post-processing) and imports nothing from the product package;
callers hand it plain arrays.

Sources, by page and section (the pages are Korean-language web articles):

* 24-ai.news, "DiffusionGemma integrated into vLLM" -- section "How does
  diffusion text generation differ?" (256-token noisy canvas; decoder mode is
  bidirectional attention inside a +-W sliding window, encoder mode is causal),
  section "Token commit mechanism" (entropy-ordered commit; self-conditioning
  by the probability-weighted embedding average).
* thakicloud.com, "DiffusionGemma-as-Jev" -- section "What is DiffusionGemma"
  (one backbone, decoder mode reads the encoder KV bidirectionally), section
  "What are Jev and structured-reads" (fixed answer positions, one parallel
  pass gives a per-alternative distribution).
* tau-home.com, "DiffusionGemma like Jev" -- section "Refusing JSON token
  generation" (prefilled canvas, blank decision slots, read the logprob and
  entropy of the allowed label ids after one denoise forward).
* sotaaz.com, "DiffusionGemma vLLM example server" -- section "The server
  accepts at most 26 alternatives per question" (A-Z labels, 422 beyond 26,
  ask_if gating, entropy > 0.1 triggers four averaged noise reads per stage,
  ``samples: 1`` pins one read).

Functions with no pin other than their own definition are marked
"parity unpinned" in their docstring; at present there are none.
"""
from .nvfp4 import (block_values, decode_e2m1, dequantize_nvfp4, from_kblock_layout,  # noqa: F401
                    from_mma_layout, pack_nibbles, quantize_nvfp4, tensor_scale, to_e2m1_codes,
                    to_kblock_layout, to_mma_layout, unpack_nibbles)
from .philox import philox4x32_10, noise_tokens, seed_key  # noqa: F401
from .quant import (dequantize_rows, e4m3_value, quantize_cols_e4m3, quantize_rows_e4m3,  # noqa: F401
                    selfcond_fp8)
from .step import (  # noqa: F401
    bf16_round,
    attn_decode,
    paged_to_contiguous,
    paged_write,
    prefill_attn,
    attn_mixed,
    lmhead_stats,
    label_logits,
    slot_noise_rows,
    slot_read,
    commit,
    selfcond_embed,
    canvas_update,
    ask_if_fires,
    ask_if_select,
    denoise_loop,
)
