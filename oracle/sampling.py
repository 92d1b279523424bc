"""Oracle sampler of the target at temperature T > 0 (test infrastructure only).

"Speculative Decoding with EAGLE", section "Technical insight": a drafted token
is accepted only when it matches the target's own choice at that point, its
argmax (greedy decoding) or its sample (sampling). At T > 0 every verified row
therefore draws the target's sample of the next token; a child of the row is
accepted when its token equals that sample, else the sample is the bonus token.
Each committed token is then a sample of the target's own next-token
distribution given the committed prefix ("yuhuili": consistency with vanilla
decoding in the distribution; "EAGLE (LLM decoding)", operational notes on the
temperature).

The sample is drawn by the Gumbel-max rule (Gumbel 1954; the softmax sampling
identity): argmax_v (logit_v / T + g_v) with g_v = -log(-log(u_v)) for
independent uniforms u_v is a sample of softmax(logit / T). The uniforms come
from a counter-based generator, SplitMix64's output function (Steele, Lea &
Flood, OOPSLA 2014), keyed by (seed, sequence, position of the sampled token,
vocabulary entry):

    k1 = mix64(seed + (seq + 1) * GAMMA)
    k2 = mix64(k1 + (pos + 1) * GAMMA)
    z  = mix64(k2 + (v + 1) * GAMMA)           GAMMA = 0x9E3779B97F4A7C15
    u  = ((z >> 40) + 0.5) * 2^-24            (exact in float32, in (0, 1))
    g  = -log(-log(u))                        (float32)

Keying by position makes the noise of position p the same wherever position p
is sampled, so speculative sampling with seed s commits exactly the tokens
that vanilla sampling with seed s commits (each committed token is the same
function of the committed prefix and the noise of its position). The CUDA
path implements the same definition in its own code; both take the argmax in
float32.

Pins (tests/test_oracle_sampling.py): mix64 against the published SplitMix64
vectors; the Gumbel-max draw against softmax(logit / T) by a chi-square test
over many keys; speculative sampling equal to vanilla sampling token for token.
"""
from __future__ import annotations

import dataclasses

import numpy as np

F32 = np.float32
GAMMA = np.uint64(0x9E3779B97F4A7C15)


def mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64's output function on uint64 values (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        return z ^ (z >> np.uint64(31))


def gumbel(seed: int, seq: int, pos: int, vocab: int) -> np.ndarray:
    """Gumbel noise g_v, v < vocab, of the token at position `pos` of sequence `seq` (float32)."""
    with np.errstate(over="ignore"):
        k1 = mix64(np.uint64(seed) + np.uint64(seq + 1) * GAMMA)
        k2 = mix64(k1 + np.uint64(pos + 1) * GAMMA)
        z = mix64(k2 + (np.arange(vocab, dtype=np.uint64) + np.uint64(1)) * GAMMA)
    u = ((z >> np.uint64(40)).astype(F32) + F32(0.5)) * F32(2.0 ** -24)
    return (-np.log(-np.log(u))).astype(F32)


@dataclasses.dataclass(frozen=True)
class Sampler:
    """The target's choice of the next token: argmax at T == 0, else the seeded Gumbel-max sample."""
    temperature: float = 0.0
    seed: int = 0

    def choose(self, logits: np.ndarray, seq: int, pos: np.ndarray) -> np.ndarray:
        """logits [rows, V] (float32); pos[r] = position of the token row r chooses. Returns int32 [rows]."""
        logits = np.asarray(logits, F32)
        if self.temperature == 0.0:
            return np.argmax(logits, axis=-1).astype(np.int32)
        T = F32(self.temperature)
        out = np.empty(logits.shape[0], np.int32)
        for r in range(logits.shape[0]):
            out[r] = np.argmax(logits[r] / T + gumbel(self.seed, seq, int(pos[r]), logits.shape[1]))
        return out

    def values(self, logits: np.ndarray, seq: int, pos: np.ndarray) -> np.ndarray:
        """The perturbed values whose argmax is the choice (logits at T == 0), for near-tie margins."""
        logits = np.asarray(logits, F32)
        if self.temperature == 0.0:
            return logits
        T = F32(self.temperature)
        return np.stack([logits[r] / T + gumbel(self.seed, seq, int(pos[r]), logits.shape[1])
                         for r in range(logits.shape[0])])


GREEDY = Sampler()
