"""Every workload at its full size, in the launch configuration the benchmark
times (automatic split count), checked on sampled (sequence, head) rows that
the oracle computes one by one (GPU only)."""
import numpy as np
import pytest

import gen
import oracle
from gpu_cases import assert_close, host, run_cuda

pytestmark = pytest.mark.gpu

FULL = ["llama3_8b", "long_70b", "mha_13b_b1", "mha_13b_b8", "mqa_13b_b1", "mqa_13b_b8",
        "sweep_bs8", "sweep_bs16", "sweep_bs32", "sweep_bs64", "sweep_bs128"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_rows(name):
    w = gen.make(name, device="cuda", poison=True)
    out, _ = run_cuda(w)
    rng = np.random.default_rng(5)
    n = min(48, w.B * w.Hq)
    flat = rng.choice(w.B * w.Hq, size=n, replace=False)
    # always include the longest and the shortest sequence
    flat = np.unique(np.concatenate([flat, [int(np.argmax(w.lens_np)) * w.Hq,
                                            int(np.argmin(w.lens_np)) * w.Hq + w.Hq - 1]]))
    rows = np.stack([flat // w.Hq, flat % w.Hq], axis=1)
    want, rc = oracle.decode_rows_f64(host(w.q), host(w.k_pool), host(w.v_pool), w.table_np,
                                      w.lens_np, w.scale, rows)
    assert rc == 0
    got = out[rows[:, 0], rows[:, 1]]
    assert_close(got, want, w.dtype, name)
    assert out.float().isfinite().all()
    del w, out
