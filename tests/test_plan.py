"""Launch plans of the scan, its backward and the SSD layer, on the CPU: ssm_scan_plan,
ssm_scan_bwd_plan and ssd_chunk_scan_plan with an explicit SM count touch no device. The
expected plans follow from the planning rules (one CTA per SM for the wide scan CTA and for the
SSD layer's chains; time segments only where the last wave or the row count leaves SMs idle;
for the backward, the segment count with the least weighted work on the most loaded SM), for a
GPU of 148 SMs."""
import torch

from selective_state_space_110_b300 import bwd_plan, scan_plan, ssd_plan

SMS = 148
STATE_BYTES = 64 * 128 * 4  # one (head, 64 x 128 fp32) SSD state


def test_scan_plan_mamba_130m_layer_runs_unsplit():
    # 8 x 1536 rows = 384 blocks of 32 channels at one row per lane: several CTAs per SM, no cut
    p = scan_plan(8, 1536, 16, 2048, sms=SMS)
    assert p == dict(rows_per_lane=1, whole_blocks=384, split_blocks=0, segments=1,
                     segment_tokens=2048, channels_per_block=32, workspace_bytes=0,
                     required_workspace_bytes=0)


def test_scan_plan_mamba_2p8b_layer_is_balanced():
    # 4 x 5120 rows = 160 wide blocks of 128 channels: 148 run whole, one per SM; the 12 left
    # over are cut into 11 segments of 192 tokens (a multiple of the 16-token chunk), so that
    # their 132 segments fill one more wave. The workspace holds each cut row's local end state
    # (16 fp32) and summed Delta for the first 10 segments; it only balances the GPU.
    p = scan_plan(4, 5120, 16, 2048, sms=SMS)
    rows = 12 * 128
    assert p == dict(rows_per_lane=2, whole_blocks=148, split_blocks=12, segments=11,
                     segment_tokens=192, channels_per_block=128,
                     workspace_bytes=rows * 10 * (64 + 4), required_workspace_bytes=0)
    assert p["segments"] * p["segment_tokens"] >= 2048 > (p["segments"] - 1) * p["segment_tokens"]


def test_scan_plan_balanced_split_needs_the_fast_path_and_the_workspace():
    unsplit = dict(rows_per_lane=2, whole_blocks=640, split_blocks=0, segments=1,
                   channels_per_block=32, workspace_bytes=0, required_workspace_bytes=0)
    for kw in (dict(in_dtype=torch.float32), dict(zoh=True), dict(workspace_bytes=0)):
        p = scan_plan(4, 5120, 16, 2048, sms=SMS, **kw)
        assert {k: p[k] for k in unsplit} == unsplit, kw
    p = scan_plan(4, 5120, 16, 2047, sms=SMS)  # seqlen % 8 != 0: the scalar tail, no wide CTA
    assert p["split_blocks"] == 0 and p["segment_tokens"] == 2047


def test_scan_plan_long_sequence_requires_its_segments():
    # 1536 rows of 1M tokens: 48 blocks of 32 channels, far fewer than the CTA slots; every
    # block is cut into 18 segments of 58,272 tokens, and the workspace is required.
    for ws in (None, 0):
        p = scan_plan(1, 1536, 16, 1 << 20, ws, sms=SMS)
        rows = 48 * 32
        need = rows * 17 * (64 + 4)
        assert p == dict(rows_per_lane=2, whole_blocks=0, split_blocks=48, segments=18,
                         segment_tokens=58272, channels_per_block=32, workspace_bytes=need,
                         required_workspace_bytes=need)
        assert 18 * 58272 >= 1 << 20 > 17 * 58272 and 58272 % 16 == 0


def test_ssd_plan_cuts_the_last_wave():
    # 4 x 80 chains on 148 SMs: 296 whole (two waves) and 24 left over; 148 // 24 = 6 segments
    # of ceil(16 / 6) = 3 chunks, workspace: local end and folded initial state of segments
    # 0-4 of each cut chain (two states each) plus their summed decays (padded to 256 bytes).
    p = ssd_plan(4, 2048, 80, sms=SMS)
    assert p == dict(whole_chains=296, cut_chains=24, segments=6, segment_chunks=3,
                     workspace_bytes=2 * 24 * 5 * STATE_BYTES + 512)
    p = ssd_plan(3, 700, 100, sms=SMS)  # 6 chunks, the last part-filled; 4 chains left over
    assert p == dict(whole_chains=296, cut_chains=4, segments=3, segment_chunks=2,
                     workspace_bytes=2 * 4 * 2 * STATE_BYTES + 256)


def test_ssd_plan_leaves_whole_waves_and_short_sequences_alone():
    for args in [(1, 2048, 80),   # 80 chains: one wave, nothing waits on a remainder
                 (2, 2048, 74),   # 148 chains: exactly one full wave
                 (4, 300, 80)]:   # 3 chunks: too short to cut
        p = ssd_plan(*args, sms=SMS)
        assert p["cut_chains"] == 0 and p["segments"] == 1 and p["workspace_bytes"] == 0, args


def test_bwd_plan_layers_run_unsplit():
    # 4 x 5120 channels: 4 x 107 CTAs of 48 channels fill the 3-per-SM slots, one wave
    p = bwd_plan(4, 5120, 16, 2048, sms=SMS)
    assert {k: p[k] for k in ("segments", "segment_tokens", "channels_per_cta", "ctas", "ctas_per_sm")} == \
        dict(segments=1, segment_tokens=2048, channels_per_cta=48, ctas=428, ctas_per_sm=3)
    # 8 x 1536: 256 CTAs, more than half the slots (no split), few enough for the 2-per-SM build
    p = bwd_plan(8, 1536, 16, 2048, sms=SMS)
    assert (p["segments"], p["ctas"], p["ctas_per_sm"]) == (1, 256, 2)


def test_bwd_plan_long_sequence_weighs_the_most_loaded_sm():
    # 1536 channels x 1M tokens: 32 blocks. 13 segments would fill the 444 slots (3 CTAs on an
    # SM, 3/13 of the sequence each), 9 put 2 CTAs on an SM (2/9, at the faster 2-per-SM rate):
    # the plan takes 9, segments of ceil(2^20 / 9) tokens rounded up to the 16-token chunk.
    p = bwd_plan(1, 1536, 16, 1 << 20, sms=SMS)
    assert {k: p[k] for k in ("segments", "segment_tokens", "ctas", "ctas_per_sm")} == \
        dict(segments=9, segment_tokens=116512, ctas=288, ctas_per_sm=2)
    assert 9 * 116512 >= 1 << 20 > 8 * 116512 and 116512 % 16 == 0
    # 48 blocks: 3 segments (1 per SM) and 9 (3 per SM) leave the same work on the most loaded
    # SM, 6 (2 per SM) less at the faster rate
    p = bwd_plan(1, 2304, 16, 1 << 20, sms=SMS)
    assert (p["segments"], p["segment_tokens"], p["ctas"], p["ctas_per_sm"]) == (6, 174768, 288, 2)


def test_bwd_plan_segments_are_at_least_4096_tokens():
    p = bwd_plan(1, 32, 16, 40000, sms=SMS)  # one block: at most 40000 // 4096 = 9 segments
    assert (p["segments"], p["segment_tokens"], p["ctas"]) == (9, 4448, 9)
    p = bwd_plan(1, 32, 16, 2048, sms=SMS)   # too short to cut
    assert (p["segments"], p["segment_tokens"]) == (1, 2048)


def test_bwd_plan_workspace_and_rejections():
    from selective_state_space_110_b300 import SelscanError
    import pytest
    full = bwd_plan(1, 1536, 16, 1 << 20, sms=SMS)["workspace_bytes"]
    given = bwd_plan(1, 1536, 16, 1 << 20, checkpoints=True, sms=SMS)["workspace_bytes"]
    # the state every 16 tokens (4 bytes per (row, token)) is the difference
    assert full - given >= 1536 * (1 << 20) * 4 and given > 0
    for kw in (dict(sms=5000), dict(sms=-1)):
        with pytest.raises(SelscanError, match="INVALID_ARG"):
            bwd_plan(1, 32, 16, 2048, **kw)
    with pytest.raises(SelscanError, match="INVALID_ARG"):
        bwd_plan(1, 32, 8, 2048, sms=SMS)
