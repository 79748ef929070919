"""CPU oracle of the CacheGen codec. TEST INFRASTRUCTURE: imported only by
the tests, the package smoke check and the bench's CPU-baseline leg."""
