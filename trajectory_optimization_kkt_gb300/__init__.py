"""GB300-native batched KKT solve for GATO-style trajectory optimisation."""
