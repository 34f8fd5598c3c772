"""CPU oracle of the CONF-KV decode step (test infrastructure only).

Only the tests, the package smoke check and the benchmark's CPU-baseline /
reference leg may import this package; the library never does.
"""
