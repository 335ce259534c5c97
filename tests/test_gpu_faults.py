"""Failure detection on the GPU without a GPU fault: bounded waits that run
out report SEP_ERR_TIMEOUT and leave the context usable; an index built for
other shapes, or inconsistent cache counters, report SEP_ERR_DEVICE_BOUNDS
and skip the work.  Nothing here traps, faults or hangs: every corrupt
input is made on the host and every kernel checks it before use."""

import numpy as np
import pytest
import torch

from separator_token_kv_sep_b300 import synth
from helpers import assert_close_rel, to_dev

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    from separator_token_kv_sep_b300 import api
    assert api.sep_get_device_status() == 0
    api.sep_selftest_wait_timeout(2000)
    assert api.sep_get_device_status() == 5  # SEP_ERR_TIMEOUT, and cleared
    assert api.sep_get_device_status() == 0
    # the context still runs real work correctly
    from oracle import sepllm as O
    q, k, v, _, ids = synth.small_prefill(1, 2, 2, 300, 64, 4, 64, 0.12, 5, "bf16", False)
    buf = api.sep_build_index(torch.from_numpy(ids).cuda(), synth.SEP_IDS, 4, 64)
    o, _ = api.sep_attn_fwd(buf, to_dev(q, torch.bfloat16), to_dev(k, torch.bfloat16),
                            to_dev(v, torch.bfloat16))
    ro, _ = O.attention_forward(q, k, v, ids, synth.SEP_IDS, 4, 64)
    assert_close_rel(o.float().cpu().numpy(), ro, what="O after timeout")
    assert api.sep_get_device_status() == 0


def test_index_for_other_shape_is_reported_not_used():
    from separator_token_kv_sep_b300 import api
    rng = np.random.default_rng(1)
    ids = synth.token_ids(rng, (1, 256), 0.1)
    buf = api.sep_build_index(torch.from_numpy(ids).cuda(), synth.SEP_IDS, 4, 64)
    # the attention call claims L = 128: the header check stops every kernel
    bf = torch.bfloat16
    q = torch.zeros((1, 2, 128, 64), dtype=bf, device="cuda")
    api.sep_attn_fwd(buf, q, q, q)
    assert api.sep_get_device_status() == 6  # SEP_ERR_DEVICE_BOUNDS
    dq, dk, dv = api.sep_attn_bwd(buf, q, q, q, q, torch.zeros((1, 2, 128), device="cuda"), q)
    assert api.sep_get_device_status() == 6
    assert api.sep_get_device_status() == 0


def test_inconsistent_cache_counters_are_reported():
    from separator_token_kv_sep_b300 import api
    S, Hkv, d, a, s, w, c = 2, 2, 64, 2, 4, 8, 20
    p = api.cache_params(S, Hkv, d, a, s, w, c)
    buf = api.sep_cache_init(p)
    # corrupt the counters of (sequence 0, kv head 0): more entries than c
    meta = buf[:32].view(torch.int32)
    meta[0] = a
    meta[3] = c + 5
    bf = torch.bfloat16
    kn = torch.zeros((S, Hkv, d), dtype=bf, device="cuda")
    qn = torch.zeros((S, 2 * Hkv, d), dtype=bf, device="cuda")
    ids = torch.zeros((S,), dtype=torch.int32, device="cuda")
    api.sep_cache_step(p, buf, qn, kn, kn, ids, synth.SEP_IDS)
    assert api.sep_get_device_status() == 6
    assert int(meta[3]) == c + 5  # the step did not write the corrupt stream


def test_keep_positions_outside_the_sequence_are_reported():
    # keep_pos entries past the row (one too far, one negative) are caught by
    # the keep-row gather and scatter before any access; the calls report
    # SEP_ERR_DEVICE_BOUNDS and the context keeps working
    from separator_token_kv_sep_b300 import api
    rng = np.random.default_rng(3)
    B, H, L, d = 2, 2, 300, 64
    ids = synth.token_ids(rng, (B, L), 0.3)
    buf = api.sep_build_index(torch.from_numpy(ids).cuda(), synth.SEP_IDS, 4, 32)
    views = api.sep_index_views(buf, B, L)
    assert int(views["keep_count"][0]) > 10 and int(views["keep_count"][1]) > 10
    views["keep_pos"][0, 5] = L + 1000
    views["keep_pos"][1, 2] = -7
    bf = torch.bfloat16
    mk = lambda *sh: torch.randn(*sh, device="cuda").to(bf)  # noqa: E731
    q, k, v, do = mk(B, H, L, d), mk(B, H, L, d), mk(B, H, L, d), mk(B, H, L, d)
    o, lse = api.sep_attn_fwd(buf, q, k, v)
    assert api.sep_get_device_status() == 6  # SEP_ERR_DEVICE_BOUNDS
    api.sep_attn_bwd(buf, q, k, v, o, lse, do)
    assert api.sep_get_device_status() == 6
    assert api.sep_get_device_status() == 0
