"""GPU index build (separator flags, keep prefix scan, compaction, block
lists) against the oracle: bit-exact."""

import numpy as np
import pytest
import torch

from oracle import sepllm as O
from separator_token_kv_sep_b300 import synth

pytestmark = pytest.mark.gpu


def run_index(ids, sep_ids, a, n):
    from separator_token_kv_sep_b300 import api
    B, L = ids.shape
    d_ids = torch.from_numpy(np.ascontiguousarray(ids, np.int32)).cuda()
    buf = api.sep_build_index(d_ids, sep_ids, a, n)
    views = {k: v.cpu().numpy() for k, v in api.sep_index_views(buf, B, L).items()}
    assert api.sep_get_device_status() == 0
    return views


def check_index(ids, sep_ids, a, n):
    B, L = ids.shape
    g = run_index(ids, sep_ids, a, n)
    kp, kpos, kc = O.keep_index(ids, sep_ids, a)
    assert np.array_equal(g["keep_prefix"], kp)
    assert np.array_equal(g["keep_count"], kc)
    for b in range(B):
        assert np.array_equal(g["keep_pos"][b, :kc[b]], kpos[b])
    assert np.array_equal(g["blocks"], O.block_list(kp, L, a, n, 128))
    assert np.array_equal(g["keep_bits"].view(np.uint32), O.separator_bitmask(ids, sep_ids, a))


@pytest.mark.parametrize("cfg", synth.PREFILL_CONFIGS, ids=lambda c: c.name)
def test_index_workloads(cfg):
    _, _, _, _, ids = synth.prefill_inputs(
        synth.PrefillConfig(cfg.name, cfg.B, 1, 1, cfg.L, 64, "f32", cfg.a, cfg.n, cfg.p,
                            cfg.seed, geometric=cfg.geometric))
    check_index(ids, synth.SEP_IDS, cfg.a, cfg.n)


@pytest.mark.parametrize("B,L,a,n,p", [
    (1, 1, 4, 1, 0.5), (3, 33, 0, 1, 0.3), (2, 127, 1, 2, 1.0), (2, 129, 4, 127, 0.0),
    (1, 4095, 4, 128, 0.12), (1, 4097, 4, 4097, 0.12), (5, 1000, 7, 100, 0.5),
    (2, 8193, 3, 1000, 0.01)])
def test_index_edge_shapes(B, L, a, n, p):
    rng = np.random.default_rng(L * 7 + n)
    ids = synth.token_ids(rng, (B, L), p)
    check_index(ids, synth.SEP_IDS, a, n)


def test_index_empty_separator_list():
    rng = np.random.default_rng(5)
    ids = synth.token_ids(rng, (2, 700), 0.3)
    check_index(ids, [], 4, 64)


def test_index_many_separator_ids():
    rng = np.random.default_rng(6)
    ids = rng.integers(0, 200, size=(2, 3000)).astype(np.int32)
    check_index(ids, list(range(100, 164)), 2, 50)


def test_index_separator_ids_sharing_table_slots():
    # ids equal modulo 1024 share a slot of the kernel's separator table;
    # tokens that land in those slots without being separators (and negative
    # ids) must still be told apart exactly
    rng = np.random.default_rng(7)
    sep = [5, 1029, 2053, -1019, 77, 77, 9000]
    pool = np.array(sep + [3077, 4101, -2043, 1101, 8999, 9001, 0, 1, 2, 1024, 2048, 5 + 4096],
                    np.int32)
    ids = pool[rng.integers(0, len(pool), size=(3, 5000))]
    check_index(ids, sep, 3, 200)


def test_index_batch64_long():
    rng = np.random.default_rng(64)
    ids = synth.token_ids(rng, (64, 65536), 0.12)
    g = run_index(ids, synth.SEP_IDS, 4, 8192)
    kp, kpos, kc = O.keep_index(ids, synth.SEP_IDS, 4)
    assert np.array_equal(g["keep_prefix"], kp)
    assert np.array_equal(g["keep_count"], kc)
