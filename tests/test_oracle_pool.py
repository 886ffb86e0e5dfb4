"""The shard-by-shard split of the oracle that the full-size GPU tests use
(tests/oracle_pool.py) gives the same per-tensor states and rows as the
oracle run on whole tensors, on a small workload (no GPU)."""
import numpy as np
import torch

import oracle_pool
import workloads


def _bits(x):
    return x.view(torch.int16).numpy().view(np.uint16)


def test_shard_split_matches_whole_tensor(orc):
    w = workloads.WORKLOADS["taco_tiny"]
    N, R, C, B = w.ranks, 64, w.cols, w.block
    gr = R // N
    x = workloads.make_rank_inputs(w, rows=R, seed=3)
    xb = _bits(x).reshape(N, R, C)
    # whole tensors: CURRENT compress, fused reduce + requant into N shards
    st = np.zeros(2 * N, dtype=np.float32)
    c, s, _ = orc.compress(orc.TACO_FP8, B, xb.reshape(-1), orc.BF16, N, R, C, st, orc.CURRENT)
    E = R * C
    shards = [(c[r * E:(r + 1) * E], s[r * E // B:(r + 1) * E // B], None, st[2 * r:2 * r + 2]) for r in range(N)]
    for fused in (True, False):
        gst = np.zeros(2 * N, dtype=np.float32)
        gst[0::2] = [0.003, 0.004, 0.002, 0.005]
        if fused:
            oc, os_, _ = orc.reduce_requant(orc.TACO_FP8, B, shards, R, C, 0, R, orc.TACO_FP8, B, N, gst,
                                            orc.DELAYED)
        else:
            ssum = orc.reduce(orc.TACO_FP8, B, shards, R, C)
            oc, os_, _ = orc.compress(orc.TACO_FP8, B, ssum, orc.FP32, N, gr, C, gst, orc.DELAYED)
        y = orc.decompress(orc.TACO_FP8, B, oc, os_, None, gst, N, gr, C, orc.BF16)
        # shard by shard
        parts = [oracle_pool.rows_amax((np.ascontiguousarray(xb[:, j * gr:(j + 1) * gr]).reshape(-1), orc.BF16,
                                        N, gr, C, B)) for j in range(N)]
        amax = np.max(np.array(parts, dtype=np.float32), axis=0)
        assert np.array_equal(amax, st[1::2])
        S1 = [orc.scale_from_amax(a) for a in amax]
        assert np.array_equal(np.array(S1, np.float32), st[0::2])
        sample = [0, 3, gr - 1]
        res = [oracle_pool.shard_chain((np.ascontiguousarray(xb[:, j * gr:(j + 1) * gr]).reshape(-1), orc.BF16, N,
                                        gr, C, orc.TACO_FP8, B, S1, orc.TACO_FP8, B, [float(gst[2 * j]), 0.0],
                                        orc.DELAYED, fused, sample, orc.BF16)) for j in range(N)]
        assert np.array_equal(np.array([v for r in res for v in r["g_state"]], np.float32), gst)
        assert np.array_equal(np.max(np.array([r["k1_amax"] for r in res], np.float32), axis=0), st[1::2])
        rows = np.array([j * gr + i for j in range(N) for i in sample])
        assert np.array_equal(np.concatenate([r["g_codes"] for r in res]), oc.reshape(R, C)[rows].reshape(-1))
        assert np.array_equal(np.concatenate([r["g_scales"] for r in res]),
                              os_.reshape(R, C // B)[rows].reshape(-1))
        assert np.array_equal(np.concatenate([r["y_rows"] for r in res]), y.reshape(R, C)[rows].reshape(-1))
        for r in range(N):
            k1c = np.concatenate([res[j]["k1_rows"][r][0] for j in range(N)])
            assert np.array_equal(k1c, c[r * E:(r + 1) * E].reshape(R, C)[rows].reshape(-1))
            k1s = np.concatenate([res[j]["k1_rows"][r][1] for j in range(N)])
            assert np.array_equal(k1s, s[r * E // B:(r + 1) * E // B].reshape(R, C // B)[rows].reshape(-1))
        if not fused:
            assert np.array_equal(np.concatenate([r["sum_rows"] for r in res]).view(np.uint32),
                                  ssum.reshape(R, C)[rows].reshape(-1).view(np.uint32))
