"""Helpers for the host replays of the kernels' barrier protocols: an mbarrier model that checks
every parity wait against the phase it names, and a random scheduler of role programs."""
import random


class Barrier:
    """mbarrier with `count` arrivals per phase; `completed` counts finished phases."""

    def __init__(self, name, count):
        self.name, self.count = name, count
        self.pending = count
        self.completed = 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, f"{self.name}: more arrivals than its count"
        if self.pending == 0:
            self.completed += 1
            self.pending = self.count

    def ready(self, parity, target):
        """A wait for completion index `target` (0-based), asked by parity as a kernel does.  The
        hardware test passes when the barrier's current phase has the other parity, so a check is
        sound only with `target` or `target + 1` phases completed: one fewer and the parity of an
        older completed phase passes it early; two more and it blocks on a phase long gone."""
        assert parity == target & 1, f"{self.name}: parity {parity} does not name completion {target}"
        assert self.completed >= target, \
            f"{self.name}: completion {target} checked after only {self.completed} completions (an older phase would pass)"
        assert self.completed <= target + 1, \
            f"{self.name}: completion {target} waited for after {self.completed} completions (aliasing)"
        return self.completed == target + 1


def wait(bar, parity, target):
    while not bar.ready(parity, target):
        yield


def run_roles(roles, seed, limit=300000):
    """Step generator programs in a random order until all finish; a long stretch with no role
    finishing is a deadlock."""
    rng = random.Random(seed)
    live = list(range(len(roles)))
    idle = 0
    while live:
        k = rng.choice(live)
        try:
            next(roles[k])
        except StopIteration:
            live.remove(k)
            idle = 0
            continue
        idle += 1
        assert idle < limit, "deadlock: no role finishes"
