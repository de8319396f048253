"""Full-size oracle results, computed on the host cores in the background.

The float64 oracle at the benchmark workloads' full sizes costs minutes of
CPU time (llama8b_32k: 8.8e12 FLOPs over every row and head).  This module
writes the exact input values once to a scratch directory and spreads
oracle.attention_rows over a pool of spawned worker processes (one BLAS
thread each), so that the oracle computes while the other GPU tests run.

A request names a workload, the query rows and the query heads to evaluate
(request_spec below).  Each request is cut into pieces of about equal work: one
query head, a run of its rows, and the key range those rows can see -- the
whole sequence when non-causal; for causal attention with documents, the
rows' own document (documents are independent: a row sees only keys of its
document, so the oracle runs on that document's slice, a decomposition that
tests/test_oracle.py checks against the whole-sequence oracle).

Worker processes are started with the "spawn" method (never forked from a
process that already uses CUDA); the inputs travel as .npy files opened with
mmap, laid out head-major so that one head's rows are contiguous (bf16 inputs
as their bit patterns, widened exactly to float32 by the worker).
"""

import multiprocessing as mp
import os
import shutil
import tempfile

import numpy as np

import workloads

# one BLAS thread per worker process: the pool supplies the parallelism
_WORKER_ENV = {"OPENBLAS_NUM_THREADS": "1", "OMP_NUM_THREADS": "1", "MKL_NUM_THREADS": "1"}
_CHUNK_ELEMS = 1 << 24  # scores per oracle chunk (128 MiB of float64)


def rotating_heads(Hq, Hkv):
    """One query head per key/value group, its position in the group
    rotating from group to group (heads 0, 5, 10, 15, 16, ... for 32/8)."""
    g = Hq // Hkv
    return [kv * g + kv % g for kv in range(Hkv)]


def request_spec(name):
    """(workload, rows or None for every row, heads) of a named request."""
    if name == "ulysses_4k":
        return "ulysses_4k", None, None
    if name == "llama8b_32k":
        return "llama8b_32k", None, None
    if name == "packed_128k":
        return "packed_128k", None, None
    if name == "halfmil_512k":       # the workload's 4096 seeded rows, every head
        cfg = workloads.CONFIGS["halfmil_512k"]
        return "halfmil_512k", workloads.sample_rows(cfg["S"], cfg["P"], cfg["sampled_rows"],
                                                     cfg["seed"], "striped"), None
    raise KeyError(name)


BACKWARD_REQUESTS = {  # name: (workload, order)
    "bwd_llama8b_32k": ("llama8b_32k", "contiguous"),
    "bwd_packed_128k_striped": ("packed_128k", "striped"),
    "bwd_halfmil_512k_striped": ("halfmil_512k", "striped"),
}
# Above this many tokens in one document, the sampled keys are only the
# sequence's last BACKWARD_TAIL_KEYS (their observers are few); a key
# further in is seen by up to S queries, whose statistics the oracle needs.
BACKWARD_TAIL_ONLY = 1 << 18
BACKWARD_TAIL_KEYS = 64
BACKWARD_DQ_ROWS = 512


def _doc_ranges(pos, S):
    """[start, end) of every document of batch row 0 (all rows of a workload
    share one position_ids row)."""
    if pos is None:
        return [(0, S)]
    starts = np.flatnonzero(np.concatenate([[1], pos[0, 1:] != pos[0, :-1] + 1]))
    ends = np.concatenate([starts[1:], [S]])
    return list(zip(starts.tolist(), ends.tolist()))


def _values(a):
    """float32 values of a stored slice: bf16 bit patterns (uint16) widen
    exactly by a 16-bit shift; float32 is returned as is."""
    if a.dtype == np.uint16:
        return (np.asarray(a).astype(np.uint32) << 16).view(np.float32)
    return np.asarray(a, dtype=np.float32)


def _rows_piece(path, h, kvh, lo, hi, rows, causal):
    """One piece in a worker: oracle.attention_rows for query head h over
    keys [lo, hi) of key/value head kvh, rows given as global indices."""
    import oracle
    qt = np.load(os.path.join(path, "q.npy"), mmap_mode="r")   # [B][Hq][S][d]
    kt = np.load(os.path.join(path, "k.npy"), mmap_mode="r")   # [B][Hkv][S][d]
    vt = np.load(os.path.join(path, "v.npy"), mmap_mode="r")
    q = _values(qt[:, h:h + 1, lo:hi]).transpose(0, 2, 1, 3)    # [B][hi-lo][1][d]
    k = _values(kt[:, kvh:kvh + 1, lo:hi]).transpose(0, 2, 1, 3)
    v = _values(vt[:, kvh:kvh + 1, lo:hi]).transpose(0, 2, 1, 3)
    pos = None
    if causal:
        pos = np.load(os.path.join(path, "pos.npy"))[:, lo:hi]
    out, lse = oracle.attention_rows(q, k, v, np.asarray(rows) - lo, pos,
                                     max_chunk_elems=_CHUNK_ELEMS)
    return out[:, :, 0, :], lse[:, 0, :]


def _load(path, name, h0, h1):
    """float32 values of heads [h0, h1) of a stored tensor, token-major
    ([B][S][h1-h0][d]) as the oracle takes them."""
    a = np.load(os.path.join(path, name + ".npy"), mmap_mode="r")  # [B][H][S][d]
    return np.ascontiguousarray(_values(a[:, h0:h1]).transpose(0, 2, 1, 3))


def _dq_piece(path, h, kvh, rows, causal):
    """dq of query head h on the given rows (oracle.attention_backward_rows)."""
    import oracle
    pos = np.load(os.path.join(path, "pos.npy")) if causal else None
    dq = oracle.attention_backward_rows(_load(path, "q", h, h + 1), _load(path, "k", kvh, kvh + 1),
                                        _load(path, "v", kvh, kvh + 1),
                                        _load(path, "dout", h, h + 1), rows, pos)
    return dq[:, :, 0, :]


def _dkdv_piece(path, h, kvh, keys, causal):
    """Query head h's share of dk, dv on the given key rows of its key/value
    head (oracle.attention_backward_keys on that head pair)."""
    import oracle
    pos = np.load(os.path.join(path, "pos.npy")) if causal else None
    dk, dv = oracle.attention_backward_keys(_load(path, "q", h, h + 1),
                                            _load(path, "k", kvh, kvh + 1),
                                            _load(path, "v", kvh, kvh + 1),
                                            _load(path, "dout", h, h + 1), keys, pos)
    return dk[:, :, 0, :], dv[:, :, 0, :]


def backward_dout(cfg, device="cuda"):
    """The upstream gradient of the full-size backward tests: N(0, 1) from a
    seeded generator (seed + 7), rounded to bf16."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(cfg["seed"] + 7)
    return torch.randn((cfg["B"], cfg["S"], cfg["Hq"], cfg["d"]), generator=g,
                       device=device).to(torch.bfloat16)


def backward_keys(pos, S, P, order):
    """Key tokens whose observers are cheap to enumerate: the last 16 tokens
    of every document, every token of documents up to 128 long, the first 16
    of documents up to 5000 long; for a single document, 48 seeded keys of
    the last block and the first 8 keys of that block -- or, for a single
    document longer than BACKWARD_TAIL_ONLY, its last BACKWARD_TAIL_KEYS
    tokens only."""
    import oracle
    seg_starts = np.nonzero(pos[0] == 0)[0]
    if len(seg_starts) == 1 and S > BACKWARD_TAIL_ONLY:
        return np.arange(S - BACKWARD_TAIL_KEYS, S, dtype=np.int64)
    ends = np.append(seg_starts[1:], S)
    keys = set()
    for a, e in zip(seg_starts, ends):
        L = e - a
        keys.update(range(max(a, e - 16), e))
        if L <= 128:
            keys.update(range(a, e))
        elif L <= 5000:
            keys.update(range(a, a + 16))
    if len(seg_starts) == 1:
        Lb = S // P
        blk = oracle.block_tokens(S, P, P - 1, order)
        rng = np.random.default_rng(S)
        keys.update(int(t) for t in rng.choice(blk, 48, replace=False))
        keys.update(range(S - Lb, S - Lb + 8))
    return np.array(sorted(keys), dtype=np.int64)


class FullSizeOracle:
    """A spawned worker pool plus the pieces of every submitted request."""

    def __init__(self, workers=None, min_piece=4096 * 4096):
        self.min_piece = float(min_piece)  # smallest piece, in (row, key) pairs
        self.dir = tempfile.mkdtemp(prefix="sp_fullsize_oracle_")
        self.workers = workers or os.cpu_count() or 1
        saved = {k: os.environ.get(k) for k in _WORKER_ENV}
        os.environ.update(_WORKER_ENV)  # inherited by the workers started now
        try:
            self.pool = mp.get_context("spawn").Pool(self.workers)
        finally:
            for k, val in saved.items():
                if val is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = val
        self.requests = {}
        self.written = set()

    def close(self):
        self.pool.terminate()
        self.pool.join()
        shutil.rmtree(self.dir, ignore_errors=True)

    def _write(self, key, q, k, v, pos):
        """Save q, k, v ([B][S][H][d]) head-major under the scratch
        directory -- numpy arrays as float32, bf16 torch tensors as their
        16-bit patterns -- and position_ids."""
        wdir = os.path.join(self.dir, key)
        os.makedirs(wdir, exist_ok=True)
        for n, t in (("q", q), ("k", k), ("v", v)):
            if isinstance(t, np.ndarray):
                a = np.ascontiguousarray(t.astype(np.float32).transpose(0, 2, 1, 3))
            else:
                import torch
                assert t.dtype == torch.bfloat16
                a = t.permute(0, 2, 1, 3).contiguous().view(torch.int16).cpu().numpy()
                a = a.view(np.uint16)
            np.save(os.path.join(wdir, n + ".npy"), a)
        if pos is not None:
            np.save(os.path.join(wdir, "pos.npy"), np.asarray(pos, dtype=np.int32))
        return wdir

    def _workload_dir(self, workload):
        """The workload's exact bf16 inputs, drawn on the GPU as the tests
        draw them (written once per workload)."""
        if workload not in self.written:
            import torch
            cfg = workloads.CONFIGS[workload]
            q, k, v = workloads.qkv_torch(cfg["B"], cfg["S"], cfg["Hq"], cfg["Hkv"], cfg["d"],
                                          cfg["seed"], torch.bfloat16, "cuda")
            self._write(workload, q, k, v, workloads.position_ids(cfg))
            del q, k, v
            self.written.add(workload)
        return os.path.join(self.dir, workload)

    def submit(self, name):
        """Queue every piece of a named request (no-op if already queued)."""
        if name in self.requests:
            return
        workload, rows, heads = request_spec(name)
        cfg = workloads.CONFIGS[workload]
        self._queue(name, self._workload_dir(workload), workloads.position_ids(cfg), rows, heads,
                    tuple(cfg[x] for x in ("B", "S", "Hq", "Hkv", "d")))

    def submit_backward(self, name):
        """Queue a backward request: dq on BACKWARD_DQ_ROWS seeded rows of
        every query head, dk and dv on backward_keys() of every key/value
        head (one piece per query head, summed over its group)."""
        if name in self.requests:
            return
        workload, order = BACKWARD_REQUESTS[name]
        cfg = workloads.CONFIGS[workload]
        B, S, Hq, Hkv, d, P = (cfg[x] for x in ("B", "S", "Hq", "Hkv", "d", "P"))
        wdir = self._workload_dir(workload)
        dpath = os.path.join(wdir, "dout.npy")
        if not os.path.exists(dpath):
            import torch
            t = backward_dout(cfg)
            np.save(dpath, t.permute(0, 2, 1, 3).contiguous().view(torch.int16).cpu().numpy()
                    .view(np.uint16))
            del t
        pos = workloads.position_ids(cfg)
        rows = workloads.sample_rows(S, P, BACKWARD_DQ_ROWS, cfg["seed"] + 3, order)
        keys = backward_keys(pos, S, P, order)
        self._queue_backward(name, wdir, pos, rows, keys, (B, Hq, Hkv, d))

    def submit_backward_arrays(self, name, q, k, v, dout, pos, rows, keys):
        """A backward request on given arrays (float32 numpy, [B][S][H][d])."""
        wdir = self._write(name, q, k, v, pos)
        np.save(os.path.join(wdir, "dout.npy"),
                np.ascontiguousarray(dout.astype(np.float32).transpose(0, 2, 1, 3)))
        self._queue_backward(name, wdir, pos, np.asarray(rows), np.asarray(keys),
                             (q.shape[0], q.shape[2], k.shape[2], q.shape[3]))

    def _queue_backward(self, name, wdir, pos, rows, keys, dims):
        B, Hq, Hkv, d = dims
        causal = pos is not None
        g = Hq // Hkv
        dq_jobs = [(h, self.pool.apply_async(_dq_piece, (wdir, h, h // g, rows, causal)))
                   for h in range(Hq)]
        kv_jobs = [(h, self.pool.apply_async(_dkdv_piece, (wdir, h, h // g, keys, causal)))
                   for h in range(Hq)]
        self.requests[name] = dict(kind="backward", rows=rows, keys=keys, dq_jobs=dq_jobs,
                                   kv_jobs=kv_jobs, dims=(B, Hq, Hkv, d), result=None)

    def backward_result(self, name, timeout=3600.0):
        """(rows, dq [B][R][Hq][d], keys, dk [B][J][Hkv][d], dv), float64."""
        self.submit_backward(name)
        req = self.requests[name]
        if req["result"] is None:
            B, Hq, Hkv, d = req["dims"]
            g = Hq // Hkv
            dq = np.zeros((B, len(req["rows"]), Hq, d))
            for h, res in req["dq_jobs"]:
                dq[:, :, h, :] = res.get(timeout)
            dk = np.zeros((B, len(req["keys"]), Hkv, d))
            dv = np.zeros_like(dk)
            for h, res in req["kv_jobs"]:
                a, b = res.get(timeout)
                dk[:, :, h // g, :] += a
                dv[:, :, h // g, :] += b
            req["result"] = (req["rows"], dq, req["keys"], dk, dv)
            req["dq_jobs"], req["kv_jobs"] = [], []
        return req["result"]

    def submit_arrays(self, name, q, k, v, pos, rows=None, heads=None):
        """Queue a request on given arrays (q [B][S][Hq][d], k/v
        [B][S][Hkv][d], pos [B][S] or None)."""
        B, S, Hq, d = q.shape
        wdir = self._write(name, q, k, v, pos)
        self._queue(name, wdir, pos, rows, heads, (B, S, Hq, k.shape[2], d))

    def _queue(self, name, wdir, pos, rows, heads, dims):
        B, S, Hq, Hkv, d = dims
        rows = np.arange(S) if rows is None else np.asarray(rows, dtype=np.int64)
        heads = list(range(Hq)) if heads is None else list(heads)
        causal = pos is not None
        if causal:
            assert (np.asarray(pos) == np.asarray(pos)[0]).all(), "one position_ids row"
        g = Hq // Hkv
        pieces = []  # (cost, head index, row index range, key range, head)
        for lo, hi in _doc_ranges(pos, S):
            a, b = np.searchsorted(rows, lo), np.searchsorted(rows, hi)
            if a == b:
                continue
            sel = rows[a:b]
            cost = (sel - lo + 1).astype(np.float64) if causal else np.full(b - a, hi - lo, float)
            target = max(float(cost.sum()) / 8.0, self.min_piece)
            edges = [0]
            acc = 0.0
            for i, c in enumerate(cost):
                acc += c
                if acc >= target and i + 1 < len(cost):
                    edges.append(i + 1)
                    acc = 0.0
            edges.append(len(cost))
            for e0, e1 in zip(edges[:-1], edges[1:]):
                kv_hi = int(sel[e1 - 1]) + 1 if causal else hi
                for hidx, h in enumerate(heads):
                    pieces.append((float(cost[e0:e1].sum()), hidx, a + e0, a + e1, lo, kv_hi, h))
        pieces.sort(key=lambda p: -p[0])  # longest first
        jobs = []
        for _, hidx, r0, r1, lo, kv_hi, h in pieces:
            res = self.pool.apply_async(_rows_piece, (wdir, h, h // g, lo, kv_hi,
                                                      rows[r0:r1], causal))
            jobs.append((res, hidx, r0, r1))
        self.requests[name] = dict(rows=rows, heads=heads, jobs=jobs,
                                   shape=(B, len(rows), len(heads), d), result=None)

    def result(self, name, timeout=3600.0):
        """(rows, heads, out [B][R][len(heads)][d], lse [B][len(heads)][R]),
        float64, waiting for the pieces still running."""
        self.submit(name)
        req = self.requests[name]
        if req["result"] is None:
            B, R, nh, d = req["shape"]
            out = np.full((B, R, nh, d), np.nan)
            lse = np.full((B, nh, R), np.nan)
            for res, hidx, r0, r1 in req["jobs"]:
                o, l_ = res.get(timeout)
                out[:, r0:r1, hidx, :] = o
                lse[:, hidx, r0:r1] = l_
            assert not np.isnan(out).any() and not np.isnan(lse).any(), name
            req["result"] = (req["rows"], req["heads"], out, lse)
            req["jobs"] = []
        return req["result"]
