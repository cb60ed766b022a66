"""Rank bodies for the two-rank tests of compensated_bit_reproducible_gb300.distributed
(spawned processes; gloo on 127.0.0.1).  Not a test module itself."""
import os
import sys

import numpy as np


def _init(rank, ws, port):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(ws)})
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    return dist


def shards(x, ws):
    """Contiguous shards in rank order (uneven: the first is the largest)."""
    cuts = [0] + [int(x.size * (r + 1) * (r + 2) / (ws * (ws + 1))) for r in range(ws)]
    cuts[-1] = x.size
    return [x[cuts[r]:cuts[r + 1]] for r in range(ws)]


class ElementOps:
    """Host stand-in for the device state calls: a "state" is a fixed-size
    byte tensor holding the elements it stands for (count, then values), and
    every value is computed by the oracle from those elements.  It checks the
    exchange protocol (gather, rank order, which states a rank merges) on the
    CPU; the device merge itself is checked against the oracle on the GPU."""
    CAP = 4096

    def __init__(self, oracle):
        self.oracle = oracle

    def _elems(self, st):
        import torch
        n = int(st[:8].view(torch.int64)[0])
        return st[8:8 + 8 * n].view(torch.float64).numpy()

    def _store(self, st, vals):
        import torch
        assert vals.size <= self.CAP
        st.zero_()
        st[:8].view(torch.int64)[0] = vals.size
        st[8:8 + 8 * vals.size].view(torch.float64)[:] = torch.from_numpy(vals.astype(np.float64))

    def state_new(self, dtype, K, device=None):
        import torch
        return torch.zeros(8 + 8 * self.CAP, dtype=torch.uint8)

    def state_deposit(self, st, x, K):
        self._store(st, np.concatenate([self._elems(st), x.numpy().astype(np.float64)]))

    def state_merge(self, dst, src, dtype, K):
        self._store(dst, np.concatenate([self._elems(dst), self._elems(src)]))

    def state_finalize(self, st, dtype, K):
        import torch
        npd = np.float32 if dtype == torch.float32 else np.float64
        return torch.tensor([self.oracle.adn_sum(self._elems(st).astype(npd), K)], dtype=dtype)

    def cumsum_from_state(self, x, st, K, out):
        import torch
        npd = x.numpy().dtype
        head = self._elems(st).astype(npd)
        full = self.oracle.adn_cumsum(np.concatenate([head, x.numpy()]), K)
        out.copy_(torch.from_numpy(full[head.size:]))
        return out


def cpu_protocol_rank(rank, ws, port, q):
    """Exchange protocol with the host stand-in: every rank's sum equals the
    oracle's sum of the whole input, and its cumulative-sum part equals the
    whole input's cumulative sum at its positions."""
    try:
        dist = _init(rank, ws, port)
        import torch
        import oracle
        from compensated_bit_reproducible_gb300 import distributed, inputs
        ops = ElementOps(oracle)
        res = {}
        for dt, K in ((np.float32, 3), (np.float64, 6)):
            x = inputs.wide_f64(3001, seed=5).astype(dt)
            mine = torch.from_numpy(shards(x, ws)[rank].copy())
            s = distributed.sum(mine, K, ops=ops)
            c = distributed.cumsum(mine, K, ops=ops)
            off = sum(p.size for p in shards(x, ws)[:rank])
            res[str(K)] = (bool(s.numpy().tobytes() == np.array([oracle.adn_sum(x, K)], dt).tobytes()),
                           bool(c.numpy().tobytes() == oracle.adn_cumsum(x, K)[off:off + mine.numel()].tobytes()))
        dist.destroy_process_group()
        q.put((rank, res))
    except Exception as e:   # reported to the parent
        q.put((rank, repr(e)))


def gpu_rank(rank, ws, port, q):
    """The device path on cuda:0 for both ranks (their kernels never wait on
    each other: the exchange is a host gather): sums and cumulative-sum parts
    against the oracle of the whole input, K = 3 and 6, float and double."""
    try:
        dist = _init(rank, ws, port)
        import torch
        import oracle
        from compensated_bit_reproducible_gb300 import distributed, inputs
        torch.cuda.set_device(0)
        res = {}
        for dt, K in ((np.float32, 3), (np.float64, 3), (np.float32, 6), (np.float64, 6)):
            x = inputs.wide_f64(300_007, seed=11).astype(dt) if dt == np.float64 else \
                inputs.normal_f32(300_007, seed=11, spikes=True)
            x = x.copy()
            x[:50_000] *= dt(1e-9)   # the index rises inside rank 1's shard for some splits
            parts = shards(x, ws)
            mine = torch.from_numpy(parts[rank].copy()).cuda()
            s = distributed.sum(mine, K).cpu().numpy()
            c = distributed.cumsum(mine, K).cpu().numpy()
            off = sum(p.size for p in parts[:rank])
            want_c = oracle.adn_cumsum_at(x, np.arange(off, off + mine.numel()), K)
            res["%s-%d" % (np.dtype(dt).name, K)] = (
                bool(s.tobytes() == np.array([oracle.adn_sum(x, K)], dt).tobytes()),
                bool(c.tobytes() == want_c.tobytes()))
        torch.cuda.synchronize()
        dist.destroy_process_group()
        q.put((rank, res))
    except Exception as e:
        q.put((rank, repr(e)))
