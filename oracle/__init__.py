"""CPU oracle for the VeriCache round: test infrastructure only (tests, smoke check, CPU baseline)."""
from .vericache import (keep_set, fp16_rne, quant_groups, pack, unpack, quant_layout,  # noqa: F401
                        quantize_kv, dequantize_kv, frag_positions, pack_block, unpack_block, attention, draft_attn, verify_attn, accept,
                        bf16_to_f32, comp_main_rows, draft_round, stagger_period, stagger_period2, stagger_phase_work, plan_stagger,
                        snapkv_votes, pool_votes, snapkv_importance, GROUP)
