"""The dispatch plan built on the GPU from a device row_ptr ([SpMM-ops] §2.1-§2.4:
packed groups, CTA rows, split rows with their segments and partial-sum slots)
must equal the host builder's plan task for task: the documented task list,
the split-row table, the uploaded device table, the counts and the statistics;
and both must equal the oracle's plan and statistics.
Cases cover long chains of groups (no long rows at all), every row long, empty
rows, tiny and extreme options, and the full 4,194,304-row power-law matrix;
bad row offsets get the host checks' error codes."""
import numpy as np
import pytest
import torch

import oracle
import synth
from csr_bsr_spmv_gb300 import spx
from gpu_util import first_rows_expected

pytestmark = pytest.mark.gpu


def _rp(lengths):
    rp = np.zeros(len(lengths) + 1, np.int32)
    rp[1:] = np.cumsum(lengths)
    return rp


def _same_plan(M, rp, opts=None):
    nnz = int(rp[-1])
    ph = spx.spx_plan_csr(M, M, nnz, rp, opts)
    pd = spx.spx_plan_csr(M, M, nnz, torch.from_numpy(rp).cuda(), opts)
    assert pd.info == ph.info
    assert pd.stats == ph.stats and pd.opts == ph.opts
    th, lh = ph.tasks()
    td, ld = pd.tasks()
    assert np.array_equal(th, td) and np.array_equal(lh, ld)
    n = ph.info["table_bytes"] // 4
    assert torch.equal(ph.table[:n].cpu(), pd.table[:n].cpu())
    assert np.array_equal(pd.device_table(), ph.device_table())
    assert np.array_equal(ph.table[:n].cpu().numpy().view(np.uint8), ph.device_table())
    # each segmented group's per-thread first rows, against a sorted search of its row offsets
    if pd.opts["lanes_div"] == 0:
        assert np.array_equal(pd.first_rows(), first_rows_expected(rp, td, pd.opts["block_nnz"]))
    # the structure fingerprint: the same on both sides, and each side validates the other's row_ptr
    assert pd.fingerprint == ph.fingerprint
    assert pd.validate(rp) == 0 and ph.validate(torch.from_numpy(rp).cuda()) == 0
    # and the oracle's plan, built from the same row offsets with the same (resolved) options
    full = oracle.plan_opts_auto(M, rp) if opts is None else dict(spx.spx_plan_opts_default(), **opts)
    assert pd.opts == full
    w = oracle.plan_spmv(M, rp, **full)
    assert np.array_equal(td, w["tasks"]) and np.array_equal(ld, w["longrows"])
    for k, v in w["counts"].items():
        assert pd.info[k] == v, k
    assert pd.stats == oracle.row_stats(M, rp)
    return ph.info


OPTS = [None,
        {"block_nnz": 1024, "lanes_div": 0},
        {"block_nnz": 2048, "block_rows": 256, "pack_max": 512, "cta_max": 8192, "seg_nnz": 4096, "lanes_div": 16},
        {"block_nnz": 64, "block_rows": 3, "pack_max": 8, "cta_max": 20, "seg_nnz": 7, "lanes_div": 2},
        {"block_nnz": 8192, "block_rows": 1024, "pack_max": 8192, "cta_max": 8192, "seg_nnz": 1, "lanes_div": 1},
        {"block_nnz": 16, "block_rows": 1, "pack_max": 0, "cta_max": 0, "seg_nnz": 5, "lanes_div": 0}]


@pytest.mark.parametrize("opts", OPTS)
@pytest.mark.parametrize("M,lmin,lmax", [(1, 0, 0), (1, 7, 7), (5, 0, 3), (1000, 0, 40), (4097, 0, 3000),
                                         (200000, 0, 12), (3000, 0, 0)])
def test_device_plan_equals_host(M, lmin, lmax, opts):
    _same_plan(M, _rp(synth.lengths_uniform(111 + M, M, lmin, lmax)), opts)


def test_device_plan_long_chain():
    """4,194,304 rows of 16 nonzeros and no long row: one run, 65,536 groups in one chain."""
    info = _same_plan(4_194_304, _rp(np.full(4_194_304, 16, np.int32)), {"block_nnz": 1024, "lanes_div": 0})
    assert info["tasks"] == 65536 and info["segmented_groups"] == 65536


def test_device_plan_power_law():
    """The power-law workload's rows (auto options): 58,846 tasks in the host plan."""
    M = 4_194_304
    lengths, _ = synth.lengths_zipf(2, M, 2.1, 200_000, 16.0)
    info = _same_plan(M, _rp(lengths))
    assert info["split_rows"] > 0 and info["cta_rows"] > 0


def test_device_plan_rejects_bad_row_ptr():
    for rp, nnz, code in [(np.array([1, 2, 3], np.int32), 3, -1),   # row_ptr[0] != 0
                          (np.array([0, 2, 3], np.int32), 4, -1),   # row_ptr[M] != nnz
                          (np.array([0, 3, 2], np.int32), 2, -3)]:  # decreasing
        with pytest.raises(spx.SpxError) as e:
            spx.spx_plan_csr(2, 2, nnz, torch.from_numpy(rp).cuda())
        assert e.value.code == code


def test_validate_detects_a_moved_entry_on_the_device():
    """Same M, K, nnz, one entry moved to the next row: the device check reports the stale plan."""
    L, _ = synth.lengths_zipf(82, 300000, 2.1, 20000, 12.0)
    rp = _rp(L)
    plan = spx.spx_plan_csr(300000, 300000, int(rp[-1]), torch.from_numpy(rp).cuda())
    moved = rp.copy()
    nz = np.flatnonzero(L > 0)
    r = int(nz[nz.size // 2])
    moved[r + 1] -= 1
    assert r + 1 < rp.size - 1 and moved[r + 1] >= moved[r]
    assert plan.validate(torch.from_numpy(moved).cuda()) == -1
    assert plan.validate(torch.from_numpy(rp).cuda()) == 0
